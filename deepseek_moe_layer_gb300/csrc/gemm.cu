// gemm.cu -- grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM),
// fed by TMA, with a per-expert tile scheduler that runs entirely on the device.
//
// Source: "Epic: Engine Inference Core Stage E - MoE + hybrid families", first paragraph
// (switch_glu over the dispatched tokens through gather_mm / gather_qmm) and
// "feat(engine): E1 DeepSeek-style MoE gate (sigmoid, group top-k, bias) (#108)", review
// section "Architecture and design" (switch_glu, then combine with the shared expert).
// Three products use the same kernel:
//   kGateUp : h[j, n] = silu(x_j . W_gate[e, n]) * (x_j . W_up[e, n])      (SwiGLU fused)
//   kDown   : o[j, c] = h_j . W_down[e, c]
//   kRouter : logits[t, e] = x_t . W_router[e]     (fp32 out, optional K split)
//
// Groups: the E routed experts (rows offsets[g] .. offsets[g+1] of the activation
// matrix) plus, optionally, the shared expert as group E (all T tokens).  A tile is
// (group, token tile, feature tile, k split); the tile list is derived on the device from
// the expert offsets, so no host synchronisation sits between dispatch and GEMM.  Tiles
// are ordered group-major, feature tile next, token tile fastest, so CTAs working at the
// same time share a weight tile through L2.
//
// Two orientations:
//   tokens on M (TOKT == 0): UMMA 128 x 256; A = 128 token rows, B = 256 weight rows
//       (kGateUp: 128 gate rows then the same 128 up rows, so one accumulator row holds
//       matching gate and up columns and the SwiGLU epilogue is thread-local).
//   tokens on N (TOKT = 16..128): UMMA 128 x TOKT; A = 128 weight rows (kGateUp: two
//       A tiles, gate and up, into two accumulators), B = TOKT token rows.  Used when the
//       experts see few tokens (decode): the weight stream is the whole cost, and putting
//       the tokens on N wastes no tensor work or shared-memory bandwidth on padding.
//
// CTA pairs (bf16 experts, tokens on M, many tokens per expert): the two CTAs of a
// cluster compute one 256 x 256 tile with cta_group::2 UMMAs issued by the even CTA.  Each
// CTA loads its own 128 token rows and half of the tile's 256 weight rows; the odd CTA's
// copies complete on the even CTA's stage barrier, the UMMAs' completion is multicast to both
// CTAs' stage and accumulator barriers, and both epilogues report to the even CTA.
//
// Warp roles (192 threads, one CTA per SM, persistent over tiles):
//   warp 0      TMA producer: a ring of kStages (activation tile, weight tile) stages;
//   warp 1      TMEM owner and UMMA issuer (one elected lane); accumulators double
//               buffered in TMEM so the epilogue of tile i overlaps the main loop of i+1;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator, SwiGLU / conversion, stores.
// Every mbarrier wait is bounded; a role that gives up records a timeout in the device
// status word, tells the others through shared memory, waits for its own copies and
// MMAs in flight, and the CTA frees its TMEM and returns.
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace moe {

__device__ unsigned int g_status;

namespace {

constexpr int kThreads = 192;
constexpr int kBK = 64;  // bf16 elements per 128-byte swizzled row = one k-block

__host__ __device__ constexpr int cmin(int a, int b) { return a < b ? a : b; }
__host__ __device__ constexpr int cmax(int a, int b) { return a > b ? a : b; }
__host__ __device__ constexpr int pow2ceil(int v) {
    int p = 1;
    while (p < v) p <<= 1;
    return p;
}

constexpr int kDequantWarps = 8;  // 4-bit variant: warps turning packed codes into bf16

template <int MODE, int TOKT, int QB, int PAIR = 0>
struct Cfg {
    static constexpr bool kQ = QB != 0;                              // affine-quantised weights
    static constexpr bool kSwap = TOKT != 0;
    // CTA pair (bf16 experts, tokens on M): the two CTAs of a cluster compute one 256 x 256
    // tile with cta_group::2 UMMAs (M = 256: 128 token rows per CTA; N = 256: each CTA loads
    // half of the weight rows), so each CTA streams 32 KB of operands per k-block instead of
    // 48 KB for the same tensor work, and six stages fit in shared memory instead of four.
    static constexpr bool kPair = PAIR != 0;
    // quantised experts with tokens on M: a tile is two 128-row token sub-tiles that share
    // every dequantised weight stage (each B tile feeds two UMMAs, one accumulator per
    // sub-tile), which halves the dequantisation work per flop.  The two accumulators fill
    // TMEM, so they are single-buffered.  (Measured: 4-bit prefill T=4096 5.18 -> 3.90 ms;
    // the bf16 experts, whose weight tiles arrive by TMA, lose more to the single-buffered
    // accumulators than they gain: 5.72 -> 6.17 ms at T=8192, so they keep 128-row tiles.)
    static constexpr bool kM2 = kQ && !kSwap && MODE != kRouter;
    static constexpr int kSub = kM2 ? 2 : 1;                         // token sub-tiles
    static constexpr int kTok = kSwap ? TOKT : 128 * kSub;           // token rows per CTA tile
    static constexpr int kTileRows = kPair ? 2 * kTok : kTok;        // token rows per tile
    static constexpr int kNW = (kSwap && MODE == kGateUp) ? 2 : 1;   // A weight tiles (swap)
    static constexpr int kWRows = kSwap ? 128 * kNW : (kPair ? 128 : 256);  // weight rows / stage
    static constexpr int kFeat = kSwap ? 128 : (MODE == kGateUp ? 128 : 256);
    static constexpr int kXBytes = kTok * 128;
    static constexpr int kWBytes = kWRows * 128;
    static constexpr int kAccCols = kSwap ? kTok * kNW : 256 * kSub;
    static constexpr int kAccBufs = kM2 ? 1 : 2;                     // accumulator buffers
    // 4-bit with tokens on N ("TMEM-A" path): the dequant warps write the bf16 weights
    // straight into TMEM (tcgen05.st) and the UMMA reads its A operand from there, so the
    // dequantised tile never crosses shared memory (which would otherwise carry 8x the HBM
    // bytes: bf16 written, then read back by the tensor core).  An operand stage is then
    // the token rows in shared memory plus kAStageCols TMEM columns of weights.
    static constexpr bool kTA = kQ && kSwap;
    static constexpr int kAStageCols = kNW * 32;  // 64 bf16 of K = 32 columns per weight tile
    static constexpr int kStageBytes = kTA ? kXBytes : kXBytes + kWBytes;  // smem per stage
    // quantised: packed codes travel in a ring of their own.  A raw slot holds kRawKB
    // k-blocks of every weight row of the tile (a 128-byte row segment, 128-byte swizzled:
    // 4 k-blocks of 4-bit codes or 2 of 8-bit codes), so each HBM access is as long as in
    // the bf16 path and the dequant warps read it without bank conflicts.  On the TMEM-A
    // path a raw slot also carries one k-block of the bf16 shared expert (the same bytes:
    // 128-byte rows).
    static constexpr int kRawKB = QB == 8 ? 2 : 4;
    static constexpr int kRBytes = kQ ? kWRows * 128 : 0;
    static constexpr int kStages =
        kTA ? cmin(8, (512 - 2 * kAccCols) / kAStageCols)
            : cmin(12, (216 * 1024 - (kQ ? 2 * kRBytes : 0)) / kStageBytes);
    static constexpr int kRawStages =
        !kQ ? 0 : kTA ? cmin(8, (216 * 1024 - kStages * kStageBytes) / kRBytes) : 2;
    static constexpr int kRawRing = kRawStages > 0 ? kRawStages : 1;  // for slot arithmetic
    static constexpr int kThreadsCta = kQ ? kThreads + 32 + 32 * kDequantWarps : kThreads;
    static constexpr int kTmemCols = kTA ? 512 : pow2ceil(cmax(32, kAccBufs * kAccCols));
    static constexpr int kN = kSwap ? kTok : 256;
    static constexpr uint32_t kIdesc = idesc_bf16(kPair ? 256 : 128, kN);
    static constexpr int kMaxGroups = 1025;
    // shared memory: operand stages | raw stages | barriers | misc | tile prefix | row offsets
    static constexpr int kRawOff = kStages * kStageBytes;
    static constexpr int kBarOff = kRawOff + kRawStages * kRBytes;
    static constexpr int kNumBars = 2 * kStages + 2 * kRawStages + 5;
    static constexpr int kMiscOff = kBarOff + 8 * kNumBars;
    static constexpr int kPrefixOff = kMiscOff + 16;
    static constexpr int kRowOffOff = kPrefixOff + 4 * (kMaxGroups + 1);
    // down with tokens on M (256 outputs per row and tile, a 2048-long main loop): each
    // epilogue warp stages 32 rows x kStgCols bf16 (4 KB: whole 128-byte lines; 2 KB on the
    // quantised paths: half lines) so that its global stores are row segments instead of one
    // 16-byte piece per row (measured: prefill down 1.99 -> 1.74 ms; the gate/up GEMM, with
    // half the outputs per tile and a 3.5x longer main loop, gained nothing)
    static constexpr int kEpiOff = (kRowOffOff + 4 * (kMaxGroups + 1) + 127) / 128 * 128;
    static constexpr int kStgCols = kQ ? 32 : 64;  // the quantised rings leave room for 8 KB
    static constexpr int kEpiBytes = (MODE == kDown && !kSwap) ? 4 * 32 * kStgCols * 2 : 0;
    static constexpr int kSmemBytes = kEpiOff + kEpiBytes + 1024;  // + align
    static_assert(kStageBytes % 1024 == 0, "stage must keep 1024-byte alignment");
    static_assert(kEpiOff % 16 == 0, "16-byte shared accesses of the staging buffer");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kN % 16 == 0 && kN >= 16 && kN <= 256, "UMMA N for M = 128");
    static_assert(!kTA || (kStages >= 2 && 2 * kAccCols + kStages * kAStageCols <= 512),
                  "TMEM budget of the TMEM-A path");
    static_assert(!kQ || kRawStages >= 2, "raw ring depth");
    static_assert(QB == 0 || QB == 4 || QB == 8, "code width");
    static_assert(!kPair || (!kQ && !kSwap && MODE != kRouter), "CTA pairs: bf16, tokens on M");
};

struct KParams {
    const int32_t* offsets;
    long long single_rows;
    int E;
    int has_shared;
    long long shared_rows;
    long long shared_act_row0;
    long long shared_out_row0;
    int Kdim;
    int F;
    int ksplit;
    long long split_stride;
    void* out;
    long long out_ld;
    // quantised weights: fp16 scale / bias per group of qgroup inputs, [rows_total,
    // Kdim / qgroup]
    const unsigned short* qscale[2];
    const unsigned short* qbias[2];
    int qgroup;  // 32, 64 or 128 (the kernel's QG)
    int q_vec;   // 8 | Kdim/qgroup and 16-byte aligned scale/bias arrays: 16-byte loads
};

// Eight packed 4-bit codes (element j in bits 4j..4j+3 of the word) -> eight bf16 weights
// w = scale * q + bias, as four bf16x2 words in element order.  Each code becomes the bf16
// number 128 + q exactly (0x43 exponent byte over the code), 128 is subtracted exactly, and
// one fused bf16x2 multiply-add applies the group's scale and bias (one rounding).
MOE_DEV uint4 dequant8(uint32_t w, uint32_t s2, uint32_t b2) {
    const uint32_t t0 = w & 0x0F0F0F0Fu;          // codes 0, 2, 4, 6, one per byte
    const uint32_t t1 = (w >> 4) & 0x0F0F0F0Fu;   // codes 1, 3, 5, 7
    const uint32_t lo = __byte_perm(t0, t1, 0x5140);  // codes 0, 1, 2, 3
    const uint32_t hi = __byte_perm(t0, t1, 0x7362);  // codes 4, 5, 6, 7
    uint32_t v[4];
    v[0] = __byte_perm(lo, 0x43u, 0x4140);  // bf16 pair (128 + c0, 128 + c1)
    v[1] = __byte_perm(lo, 0x43u, 0x4342);
    v[2] = __byte_perm(hi, 0x43u, 0x4140);
    v[3] = __byte_perm(hi, 0x43u, 0x4342);
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t q;
        asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(q) : "r"(v[i]), "r"(0x43004300u));
        asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r[i]) : "r"(q), "r"(s2), "r"(b2));
    }
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// Eight packed 8-bit codes (element j in bits 8j..8j+7 of w0 for j < 4, of w1 for j >= 4)
// -> eight bf16 weights w = scale * q + bias.  Each code becomes the fp32 number 2^23 + q
// exactly (0x4B exponent byte over the code), 2^23 is subtracted exactly, one fp32 fused
// multiply-add applies scale and bias, and the pair is rounded once to bf16x2.
MOE_DEV uint4 dequant8_u8(uint32_t w0, uint32_t w1, float sc, float bi) {
    float q[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        q[e] = __uint_as_float(__byte_perm(w0, 0x4B000000u, 0x7440u | (uint32_t)e)) - 8388608.0f;
        q[4 + e] = __uint_as_float(__byte_perm(w1, 0x4B000000u, 0x7440u | (uint32_t)e)) - 8388608.0f;
    }
    uint32_t r[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        r[i] = pack_bf16x2(fmaf(sc, q[2 * i], bi), fmaf(sc, q[2 * i + 1], bi));
    return make_uint4(r[0], r[1], r[2], r[3]);
}

// The GPS consecutive 16-bit values of an 8-value window v that start at `off` (a multiple
// of GPS), two per word: values 2i and 2i+1 in the low and high half of out[i].
template <int GPS>
MOE_DEV void window_part(const uint4& v, int off, uint32_t (&out)[(GPS + 1) / 2]) {
    if constexpr (GPS == 8) {
        out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
    } else if constexpr (GPS == 4) {
        const bool h = off >= 4;
        out[0] = h ? v.z : v.x;
        out[1] = h ? v.w : v.y;
    } else if constexpr (GPS == 2) {
        const int q = off >> 1;
        out[0] = q == 0 ? v.x : q == 1 ? v.y : q == 2 ? v.z : v.w;
    } else {
        const uint32_t w = off < 2 ? v.x : off < 4 ? v.y : off < 6 ? v.z : v.w;
        out[0] = (off & 1) ? (w >> 16) : (w & 0xFFFFu);
    }
}

// Staged epilogue stores.  A warp's 32 accumulator rows (one per lane) are written to a
// shared buffer of 32 rows x COLS bf16 as 16-byte chunks, then read back with COLS/8 lanes per
// row so that each warp store covers whole row segments (a 128-byte line for 64 columns, half
// a line for 32).  The chunk index is XOR-swizzled with the row so that both the row-per-lane
// writes and the segment-per-lanes reads are free of bank conflicts.
template <int COLS>
MOE_DEV int stage_chunk(int r, int j) {
    return COLS == 64 ? (j ^ (r & 7)) : (j ^ ((r >> 1) & 3));
}
template <int COLS>
MOE_DEV void stage_put(uint8_t* stg, int r, int j, uint4 v) {
    *reinterpret_cast<uint4*>(stg + r * (COLS * 2) + (stage_chunk<COLS>(r, j) << 4)) = v;
}
// Row rr (< 32) of the staging buffer goes to out[row0 + rr][col0 + 8j .. +7] when the row
// is one of the tile's `rows` valid ones (rr + rbase < rows) and the columns lie below F.
template <int COLS>
MOE_DEV void staged_store(const uint8_t* stg, int lane, __nv_bfloat16_raw* out, long long row0,
                          long long ld, int col0, int rbase, int rows, int F) {
    constexpr int kCh = COLS / 8;        // 16-byte chunks per staged row
    constexpr int kRowsPer = 32 / kCh;   // rows per warp store
    const int j = lane % kCh;
    const bool cvalid = col0 + 8 * j + 8 <= F;  // F is a multiple of 8
#pragma unroll
    for (int it = 0; it < kCh; ++it) {
        const int rr = it * kRowsPer + lane / kCh;
        const uint4 w = *reinterpret_cast<const uint4*>(stg + rr * (COLS * 2) +
                                                         (stage_chunk<COLS>(rr, j) << 4));
        if (rbase + rr < rows && cvalid)
            *reinterpret_cast<uint4*>(out + (row0 + rr) * ld + col0 + 8 * j) = w;
    }
}

MOE_DEV void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct TileInfo {
    int g;               // group (E = shared)
    bool shared;
    long long act_row;   // first activation row of the tile
    long long out_row;   // first output row of the tile
    int rows;            // valid token rows in the tile
    int f;               // feature tile
    int kb0, kb1;        // k-block range
    int ks;              // k split
};

// Tiles of group g: ceil(rows_g / kTok) token tiles x feature tiles x k splits.
template <class C>
MOE_DEV int group_tiles(long long rows, int ftiles, int ksplit) {
    return (int)((rows + C::kTileRows - 1) / C::kTileRows) * ftiles * ksplit;
}

template <class C>
MOE_DEV long long group_rows(const KParams& p, const int32_t* rowoff, int g) {
    if (!p.offsets) return p.single_rows;
    if (g == p.E) return p.shared_rows;
    return (long long)(rowoff[g + 1] - rowoff[g]);
}

// Tile t of the tile list.  For a CTA pair, `rank` picks this CTA's 128 token rows of the
// pair's 256 (rows may then be 0: the peer's half of a short tile).
template <class C>
MOE_DEV TileInfo decode_tile(const KParams& p, const int32_t* prefix, const int32_t* rowoff,
                             int ngroups, int t, int rank = 0) {
    // largest g with prefix[g] <= t (empty groups repeat the prefix and are skipped)
    int lo = 0, hi = ngroups - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
    }
    TileInfo ti;
    ti.g = lo;
    ti.shared = p.offsets && lo == p.E;
    const long long rows = group_rows<C>(p, rowoff, lo);
    const int mt = (int)((rows + C::kTileRows - 1) / C::kTileRows);
    const int ft = (p.F + C::kFeat - 1) / C::kFeat;
    int local = t - prefix[lo];
    const int m = local % mt;
    local /= mt;
    ti.f = local % ft;
    ti.ks = local / ft;
    const long long r0 = (long long)m * C::kTileRows + (long long)rank * C::kTok;
    const long long left = rows - r0;
    ti.rows = (int)(left < 0 ? 0 : (left < C::kTok ? left : C::kTok));
    if (ti.shared) {
        ti.act_row = p.shared_act_row0 + r0;
        ti.out_row = p.shared_out_row0 + r0;
    } else {
        const long long base = p.offsets ? (long long)rowoff[lo] : 0;
        ti.act_row = base + r0;
        ti.out_row = base + r0;
    }
    const int nkb = p.Kdim / kBK / p.ksplit;
    ti.kb0 = ti.ks * nkb;
    ti.kb1 = ti.kb0 + nkb;
    return ti;
}

MOE_DEV void record_timeout(volatile int* abort) {
    *abort = 1;
    atomicCAS(&g_status, 0u, kStatusTimeout);
}

// tm_w0 / tm_w1: bf16 weight rows (Q4 = false) or packed 4-bit code rows (Q4 = true); the
// shared expert's maps tm_sw0 / tm_sw1 are always bf16.
template <int MODE, int TOKT, int QB, int QG, int PAIR>
__global__ void __launch_bounds__(Cfg<MODE, TOKT, QB, PAIR>::kThreadsCta, 1)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_act,
                    const __grid_constant__ CUtensorMap tm_act_sh,
                    const __grid_constant__ CUtensorMap tm_w0,
                    const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_sw0,
                    const __grid_constant__ CUtensorMap tm_sw1, const KParams p) {
    using C = Cfg<MODE, TOKT, QB, PAIR>;
    constexpr bool Q4 = C::kQ;  // any affine-quantised width (4 or 8 bits)
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
    uint64_t* full = bars;
    uint64_t* empty = bars + C::kStages;
    uint64_t* rawfull = bars + 2 * C::kStages;            // 4-bit: codes of a raw slot landed
    uint64_t* rawempty = rawfull + C::kRawStages;         // 4-bit: raw slot read, reusable
    uint64_t* tfull = rawempty + C::kRawStages;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tfull + 4;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kMiscOff + 4);
    int32_t* prefix = reinterpret_cast<int32_t*>(smem + C::kPrefixOff);
    int32_t* rowoff = reinterpret_cast<int32_t*>(smem + C::kRowOffOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = p.offsets ? p.E + p.has_shared : 1;
    const int ftiles = (p.F + C::kFeat - 1) / C::kFeat;
    // CTA pair: rank 0 (the leader) issues the pair's UMMAs; both CTAs walk the same tiles
    const int crank = C::kPair ? (int)cluster_rank() : 0;
    const bool leader = crank == 0;
    const int tstart = C::kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int tstep = C::kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    // ---- set-up: barriers, TMEM, group offsets and the tile prefix ----
    // (barriers, TMEM and the tensor maps touch nothing the kernel before writes: with a
    // programmatic launch this overlaps that kernel's tail; pdl_wait() comes before the first
    // read of its results)
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            // a pair's stage s completes on the leader's full[s]: the leader's arrival
            // expects the bytes of both CTAs' copies
            mbar_init(&full[s], Q4 ? 1 + kDequantWarps : 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < C::kRawStages; ++s) {
            mbar_init(&rawfull[s], 1);
            mbar_init(&rawempty[s], kDequantWarps);
        }
        mbar_init(&tfull[0], 1);
        mbar_init(&tfull[1], 1);
        // pair: one arrival per epilogue warp of both CTAs (on the leader's barrier)
        mbar_init(&tempty[0], C::kPair ? 8 : 128);
        mbar_init(&tempty[1], C::kPair ? 8 : 128);
        mbar_init(done, 1);
        *abort = 0;
        fence_mbar_init();
        prefetch_tmap(&tm_act);
        prefetch_tmap(&tm_act_sh);
        prefetch_tmap(&tm_w0);
        prefetch_tmap(&tm_w1);
        prefetch_tmap(&tm_sw0);
        prefetch_tmap(&tm_sw1);
    }
    if (warp == 1) {
        if constexpr (C::kPair) tmem_alloc_pair(tmem_slot, C::kTmemCols);
        else tmem_alloc(tmem_slot, C::kTmemCols);
    }
    pdl_wait();
    if (p.offsets)
        for (int i = threadIdx.x; i <= p.E; i += blockDim.x) rowoff[i] = p.offsets[i];
    __syncthreads();
    if (warp == 0) {
        const int per = (ngroups + 31) / 32;
        const int g0 = lane * per, g1 = min(ngroups, g0 + per);
        int local = 0;
        for (int g = g0; g < g1; ++g)
            local += group_tiles<C>(group_rows<C>(p, rowoff, g), ftiles, p.ksplit);
        int incl = local;
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += v;
        }
        int run = incl - local;
        for (int g = g0; g < g1; ++g) {
            prefix[g] = run;
            run += group_tiles<C>(group_rows<C>(p, rowoff, g), ftiles, p.ksplit);
        }
        if (lane == 31) prefix[ngroups] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    int total = prefix[ngroups];
    if constexpr (C::kPair) {
        // the peer's barriers are initialised and its TMEM allocated beyond this point; the
        // pair's UMMAs address the same columns in both CTAs, so both must hold them
        cluster_sync();
        if (ld_shared_cluster_u32(mapa_shared(tmem_slot, (uint32_t)(crank ^ 1))) != tmem_base) {
            total = 0;
            if (threadIdx.x == 0) atomicCAS(&g_status, 0u, kStatusPairTmem);
        }
    }

    if (warp == 0) {
        // =============================== TMA producer ===============================
        if (lane == 0) {
            // L2 policies: with tokens on N (small batches) a weight tile is read once and is
            // streamed evict-first; with tokens on M it is read by every token tile of its
            // expert, CTAs that run at the same time but drift apart along K, so it is kept
            // (evict-last, like the token rows: prefill T=8192 gate/up 3.27 -> 3.10 ms, DRAM
            // traffic of the launch 12.6 -> see the bench's traffic table)
            const uint64_t pol_w = C::kSwap ? policy_evict_first() : policy_evict_last();
            const uint64_t pol_x = policy_evict_last();
            int it = 0, s = 0;  // k-blocks issued; ring stage and its phase
            uint32_t ph = 0u;
            bool ok = true;
            for (int t = tstart; t < total && ok; t += tstep) {
                const TileInfo ti = decode_tile<C>(p, prefix, rowoff, ngroups, t, crank);
                const CUtensorMap* am = ti.shared ? &tm_act_sh : &tm_act;
                const CUtensorMap* w0 = ti.shared ? &tm_sw0 : &tm_w0;
                const CUtensorMap* w1 = ti.shared ? &tm_sw1 : &tm_w1;
                const int wrow = (ti.shared || !p.offsets ? 0 : ti.g * p.F) + ti.f * C::kFeat;
                for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++it) {
                    if (it > 0 && ++s == C::kStages) { s = 0; ph ^= 1u; }
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort)) { record_timeout(abort); ok = false; break; }
                    uint8_t* st = smem + s * C::kStageBytes;
                    const int kx = kb * kBK;
                    uint8_t* wst = st + C::kXBytes;
                    if (C::kTA || (Q4 && !ti.shared)) {
                        // token rows only: the dequant warps fill the weight tile (TMEM on
                        // the TMEM-A path, else shared memory) and complete full[s]
                        mbar_arrive_expect_tx(&full[s], C::kXBytes);
                        tma_load_2d(st, am, &full[s], kx, (int)ti.act_row, pol_x);
                        continue;
                    }
                    if (C::kPair) {
                        // this CTA's token rows and its half of the pair's 256 weight rows
                        // (gate rows in the leader, up rows in the peer, or the first /
                        // second 128 down rows), both completing on the leader's full[s]
                        const int wr = MODE == kGateUp ? wrow : wrow + crank * 128;
                        const CUtensorMap* wm = (MODE == kGateUp && crank) ? w1 : w0;
                        if (leader) {
                            mbar_arrive_expect_tx(&full[s], 2 * (C::kXBytes + C::kWBytes));
                            tma_load_2d(st, am, &full[s], kx, (int)ti.act_row, pol_x);
                            tma_load_2d(wst, wm, &full[s], kx, wr, pol_w);
                        } else {
                            const uint32_t lb = mapa_shared(&full[s], 0);
                            tma_load_2d_pair(st, am, lb, kx, (int)ti.act_row, pol_x);
                            tma_load_2d_pair(wst, wm, lb, kx, wr, pol_w);
                        }
                        continue;
                    }
                    mbar_arrive_expect_tx(&full[s], C::kXBytes + C::kWBytes);
                    tma_load_2d(st, am, &full[s], kx, (int)ti.act_row, pol_x);
                    if (MODE == kGateUp) {
                        tma_load_2d(wst, w0, &full[s], kx, wrow, pol_w);
                        tma_load_2d(wst + 128 * 128, w1, &full[s], kx, wrow, pol_w);
                    } else {
                        tma_load_2d(wst, w0, &full[s], kx, wrow, pol_w);
                    }
                }
            }
            if (!ok && leader) {
                // let the copies already issued land before the CTA can exit (full[s] also
                // waits for the dequant warps in the 4-bit case, and for the peer's copies in
                // a pair: bounded, then give up)
                for (int n = (it > C::kStages ? it - C::kStages : 0); n < it; ++n)
                    mbar_wait(&full[n % C::kStages], (uint32_t)(n / C::kStages) & 1u, nullptr,
                              100000000ull);
            }
        }
    } else if (Q4 && warp == kThreads / 32) {
        // ======================= 4-bit: packed-code TMA producer =====================
        // runs up to kRawStages k-blocks ahead of the dequant warps, independent of the
        // operand ring, so enough HBM reads stay in flight to stream the codes at full rate
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first();
            int rit = 0, rs = 0;  // raw slots issued; raw ring slot and its phase
            uint32_t rph = 0u;
            bool ok = true;
            for (int t = tstart; t < total && ok; t += tstep) {
                const TileInfo ti = decode_tile<C>(p, prefix, rowoff, ngroups, t, crank);
                if (ti.shared) {
                    // normal-mode 4-bit: the operand producer loads the bf16 shared rows;
                    // TMEM-A path: one k-block of them per raw slot (same 128-byte rows)
                    if constexpr (C::kTA) {
                        for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++rit) {
                            if (rit > 0 && ++rs == C::kRawRing) { rs = 0; rph ^= 1u; }
                            if (!mbar_wait(&rawempty[rs], rph ^ 1u, abort)) { record_timeout(abort); ok = false; break; }
                            uint8_t* rst = smem + C::kRawOff + rs * C::kRBytes;
                            mbar_arrive_expect_tx(&rawfull[rs], C::kRBytes);
                            tma_load_2d(rst, &tm_sw0, &rawfull[rs], kb * kBK, ti.f * C::kFeat, pol_w);
                            if (MODE == kGateUp)
                                tma_load_2d(rst + 128 * 128, &tm_sw1, &rawfull[rs], kb * kBK,
                                            ti.f * C::kFeat, pol_w);
                        }
                    }
                    continue;
                }
                const int wrow = ti.g * p.F + ti.f * C::kFeat;
                for (int kb = ti.kb0; kb < ti.kb1; kb += C::kRawKB, ++rit) {
                    if (rit > 0 && ++rs == C::kRawRing) { rs = 0; rph ^= 1u; }
                    if (!mbar_wait(&rawempty[rs], rph ^ 1u, abort)) { record_timeout(abort); ok = false; break; }
                    uint8_t* rst = smem + C::kRawOff + rs * C::kRBytes;
                    mbar_arrive_expect_tx(&rawfull[rs], C::kRBytes);
                    const int wx = kb * 2 * QB;  // first code word of k-block kb
                    if (MODE == kGateUp) {
                        tma_load_2d(rst, &tm_w0, &rawfull[rs], wx, wrow, pol_w);
                        tma_load_2d(rst + 128 * 128, &tm_w1, &rawfull[rs], wx, wrow, pol_w);
                    } else {
                        tma_load_2d(rst, &tm_w0, &rawfull[rs], wx, wrow, pol_w);
                    }
                }
            }
            if (!ok) {
                for (int n = (rit > C::kRawStages ? rit - C::kRawStages : 0); n < rit; ++n)
                    mbar_wait(&rawfull[n % C::kRawRing], (uint32_t)(n / C::kRawRing) & 1u,
                              nullptr, 100000000ull);
            }
        }
    } else if (warp == 1 && C::kPair && !leader) {
        // pair peer: the leader's thread issues the pair's UMMAs
    } else if (warp == 1) {
        // ================================ UMMA issuer ===============================
        if (lane == 0) {
            int it = 0, lt = 0, s = 0;  // k-blocks consumed; ring stage and its phase
            uint32_t ph = 0u;
            bool ok = true;
            for (int t = tstart; t < total && ok; t += tstep, ++lt) {
                const TileInfo ti = decode_tile<C>(p, prefix, rowoff, ngroups, t, crank);
                const int ab = C::kAccBufs == 2 ? (lt & 1) : 0;
                const uint32_t aph = (uint32_t)(C::kAccBufs == 2 ? (lt >> 1) : lt) & 1u;
                if (!(C::kPair ? mbar_wait_cluster(&tempty[ab], aph ^ 1u, abort)
                               : mbar_wait(&tempty[ab], aph ^ 1u, abort))) { record_timeout(abort); break; }
                tc_fence_after();
                const uint32_t acc = tmem_base + (uint32_t)(ab * C::kAccCols);
                for (int kb = ti.kb0; kb < ti.kb1; ++kb, ++it) {
                    if (it > 0 && ++s == C::kStages) { s = 0; ph ^= 1u; }
                    if (!(C::kPair ? mbar_wait_cluster(&full[s], ph, abort)
                                   : mbar_wait(&full[s], ph, abort))) { record_timeout(abort); ok = false; break; }
                    tc_fence_after();
                    const uint32_t xs = smem_u32(smem + s * C::kStageBytes);
                    const uint32_t ws = xs + C::kXBytes;
                    // the stage's operand descriptors, once; a K = 16 step is 32 bytes further
                    // (2 in the address field, which holds any shared-memory address)
                    const uint64_t dx = sdesc_k128(xs), dw = sdesc_k128(ws);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint32_t accum = (kb > ti.kb0 || kk > 0) ? 1u : 0u;
                        const uint64_t dxk = dx + (uint64_t)(2 * kk), dwk = dw + (uint64_t)(2 * kk);
                        if (C::kTA) {
                            // A (weights) from this stage's TMEM columns, 8 per K=16 slice
                            const uint32_t a0 = tmem_base + (uint32_t)(2 * C::kAccCols +
                                                                       s * C::kAStageCols + kk * 8);
#pragma unroll
                            for (int w = 0; w < C::kNW; ++w)
                                umma_bf16_ta(acc + (uint32_t)(w * C::kTok),
                                             a0 + (uint32_t)(w * 32), dxk, C::kIdesc, accum);
                        } else if (C::kSwap) {
#pragma unroll
                            for (int w = 0; w < C::kNW; ++w)
                                umma_bf16(acc + (uint32_t)(w * C::kTok),
                                          dwk + (uint64_t)(w * 128 * 128 / 16), dxk, C::kIdesc, accum);
                        } else if (C::kPair) {
                            umma_bf16_pair(acc, dxk, dwk, C::kIdesc, accum);
                        } else {
                            umma_bf16(acc, dxk, dwk, C::kIdesc, accum);
                            // the second sub-tile's tokens, when the tile has any
                            if (C::kM2 && ti.rows > 128)
                                umma_bf16(acc + 256u, dxk + (uint64_t)(128 * 128 / 16), dwk,
                                          C::kIdesc, accum);
                        }
                    }
                    if (C::kPair) umma_commit_pair(&empty[s], 3);  // both CTAs' stage s
                    else umma_commit(&empty[s]);
                }
                if (!ok) break;
                if (C::kPair) umma_commit_pair(&tfull[ab], 3);
                else umma_commit(&tfull[ab]);
            }
            // drain every UMMA issued by this thread before TMEM can be released
            if (it > 0) {
                if (C::kPair) umma_commit_pair(done, 1);
                else umma_commit(done);
                mbar_wait(done, 0u, nullptr, 100000000ull);
            }
        }
    } else if (Q4 && warp >= kThreads / 32) {
        // ============================ 4-bit dequantisation ==========================
        // 256 threads; thread dt owns row dt % kWRows of the stage's weight tile and
        // kWordsPT of its 8 packed words (one 64-element k-block = one scale group).
        // On the TMEM-A path a warp may only write its own TMEM lane quarter, so the row
        // follows the warp: quarter q = warp % 4, lane -> row q*32 + lane; the two warps of a
        // quarter take the gate and the up tile (gate/up) or the two halves of a row (down).
        constexpr int kWordsPT = C::kWRows * 8 / (32 * kDequantWarps);  // 8-code chunks
        constexpr int kWPC = QB >= 4 ? QB / 4 : 1;   // code words per chunk (1 or 2)
        constexpr int kPieces = kWordsPT * kWPC / 4;  // 16-byte pieces of codes per k-block
        static_assert(!Q4 || kPieces >= 1, "whole 16-byte pieces of codes per thread");
        const int dt = threadIdx.x - kThreads - 32;
        const int qtr = warp & 3;
        const int half = dt / (32 * kDequantWarps / 2);
        const int r = C::kTA ? (MODE == kGateUp ? half * 128 : 0) + qtr * 32 + lane
                             : dt % C::kWRows;
        const int wd0 = C::kTA ? (MODE == kGateUp ? 0 : half * kWordsPT)
                               : (dt / C::kWRows) * kWordsPT;
        const int mat = (MODE == kGateUp && r >= 128) ? 1 : 0;
        const int rr = (MODE == kGateUp) ? (r & 127) : r;
        const unsigned short* sp = mat ? p.qscale[1] : p.qscale[0];
        const unsigned short* bp = mat ? p.qbias[1] : p.qbias[0];
        constexpr int qsh = QG == 32 ? 5 : (QG == 128 ? 7 : 6);  // log2 inputs per group
        const int ngr = p.Kdim >> qsh;  // scale groups per row
        // scale/bias of a row are contiguous over its groups: with 8 | ngr (and 16-byte
        // aligned arrays) they arrive 8 groups per 16-byte load into a sliding window of two
        // loads (the next one in flight while the current is used); otherwise per k-block.
        const bool vec = p.q_vec != 0;
        auto pick16 = [](const uint4& v, int j) -> unsigned short {
            const uint32_t w = j < 2 ? v.x : j < 4 ? v.y : j < 6 ? v.z : v.w;
            return (unsigned short)((j & 1) ? (w >> 16) : (w & 0xFFFFu));
        };
        // ring positions, advanced once per k-block (operand stage s, phase ph) and once per
        // raw slot (rs, rph) in the order the producers and the MMA thread use them
        int s = 0, rs = 0;
        uint32_t ph = 0u, rph = 0u;
        bool ok = true;
        for (int t = tstart; t < total && ok; t += tstep) {
            const TileInfo ti = decode_tile<C>(p, prefix, rowoff, ngroups, t, crank);
            const uint32_t tcol0 = tmem_base + ((uint32_t)(qtr * 32) << 16) +
                                   (uint32_t)(2 * C::kAccCols + (MODE == kGateUp ? half * 32 : 0) +
                                              wd0 * 4);
            if (ti.shared) {
                // bf16 shared expert: its weight tile comes by TMA (normal path) or, on the
                // TMEM-A path, one k-block per raw slot whose 128-byte rows are already the
                // operand
                for (int kb = ti.kb0; kb < ti.kb1; ++kb) {
                    uint4 bw[kWordsPT];
                    if constexpr (C::kTA) {
                        if (!mbar_wait(&rawfull[rs], rph, abort)) { record_timeout(abort); ok = false; break; }
                        const uint8_t* rrow = smem + C::kRawOff + rs * C::kRBytes + r * 128;
#pragma unroll
                        for (int w = 0; w < kWordsPT; ++w)
                            bw[w] = *reinterpret_cast<const uint4*>(rrow + (((wd0 + w) ^ (r & 7)) << 4));
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&rawempty[rs]);
                        if (++rs == C::kRawRing) { rs = 0; rph ^= 1u; }
                    }
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort)) { record_timeout(abort); ok = false; break; }
                    if constexpr (C::kTA) {
                        tc_fence_after();
                        const uint32_t tcol = tcol0 + (uint32_t)(s * C::kAStageCols);
#pragma unroll
                        for (int h = 0; h < kWordsPT / 4; ++h) {
                            uint32_t v16[16];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v16[4 * i] = bw[4 * h + i].x; v16[4 * i + 1] = bw[4 * h + i].y;
                                v16[4 * i + 2] = bw[4 * h + i].z; v16[4 * i + 3] = bw[4 * h + i].w;
                            }
                            tmem_st16(tcol + (uint32_t)(16 * h), v16);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                    } else {
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[s]);
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
                continue;
            }
            const bool rvalid = ti.f * C::kFeat + rr < p.F;
            const long long grow = (long long)ti.g * p.F + ti.f * C::kFeat + rr;
            const unsigned short* srow = sp + grow * ngr;
            const unsigned short* brow = bp + grow * ngr;
            uint4 sc_cur = make_uint4(0, 0, 0, 0), bc_cur = sc_cur, sc_nxt = sc_cur, bc_nxt = sc_cur;
            int wb = ((ti.kb0 * kBK) >> qsh) & ~7;  // first group of the window (multiple of 8)
            if (rvalid && vec) {
                sc_cur = __ldg(reinterpret_cast<const uint4*>(srow + wb));
                bc_cur = __ldg(reinterpret_cast<const uint4*>(brow + wb));
                if (wb + 8 < ngr) {
                    sc_nxt = __ldg(reinterpret_cast<const uint4*>(srow + wb + 8));
                    bc_nxt = __ldg(reinterpret_cast<const uint4*>(brow + wb + 8));
                }
            }
            // one raw slot (kRawKB k-blocks of this row's codes) per pass; the k-block within
            // the slot is known at compile time.  When the thread's chunks start its rows'
            // k-blocks and the tile starts on a slot boundary, a slot's groups are a fixed part
            // of the 8-group scale window, taken once per slot; each k-block then reads its
            // group's scale and bias at a compile-time position.
            constexpr int kGPS = QG ? C::kRawKB * kBK / QG : 1;  // scale groups per raw slot
            const bool slot_win = vec && wd0 == 0 && ti.kb0 % C::kRawKB == 0;
            for (int kbs = ti.kb0; kbs < ti.kb1 && ok; kbs += C::kRawKB) {
                if (!mbar_wait(&rawfull[rs], rph, abort)) { record_timeout(abort); ok = false; break; }
                const uint8_t* rrow = smem + C::kRawOff + rs * C::kRBytes + r * 128;
                uint32_t sgw[(kGPS + 1) / 2], bgw[(kGPS + 1) / 2];
                if (slot_win) {
                    const int gs = (kbs * kBK) >> qsh;
                    if (gs >= wb + 8) {  // slots advance by kGPS groups, which divides 8
                        sc_cur = sc_nxt;
                        bc_cur = bc_nxt;
                        wb += 8;
                        if (rvalid && wb + 8 < ngr) {
                            sc_nxt = __ldg(reinterpret_cast<const uint4*>(srow + wb + 8));
                            bc_nxt = __ldg(reinterpret_cast<const uint4*>(brow + wb + 8));
                        }
                    }
                    window_part<kGPS>(sc_cur, gs - wb, sgw);
                    window_part<kGPS>(bc_cur, gs - wb, bgw);
                }
#pragma unroll
                for (int j = 0; j < C::kRawKB; ++j) {
                    const int kb = kbs + j;
                    if (kb >= ti.kb1) break;
                    // the (at most two) groups of this thread's chunks in k-block kb
                    const int e0 = kb * kBK + 8 * wd0;
                    const int ga = e0 >> qsh, gb = (e0 + 8 * kWordsPT - 1) >> qsh;
                    unsigned short sa = 0, ba = 0, sb = 0, bb = 0;  // fp16 bits
                    if (slot_win) {
                        // groups j*kBK/QG and (j*kBK + kBK-1)/QG of the slot
                        const int ia = QG ? (j * kBK) / QG : 0;
                        const int ib = QG ? (j * kBK + kBK - 1) / QG : 0;
                        sa = (unsigned short)(sgw[ia / 2] >> (16 * (ia & 1)));
                        ba = (unsigned short)(bgw[ia / 2] >> (16 * (ia & 1)));
                        sb = (unsigned short)(sgw[ib / 2] >> (16 * (ib & 1)));
                        bb = (unsigned short)(bgw[ib / 2] >> (16 * (ib & 1)));
                    } else if (vec) {
                        if (ga >= wb + 8) {  // the groups advance by at most 2 per k-block
                            sc_cur = sc_nxt;
                            bc_cur = bc_nxt;
                            wb += 8;
                            if (rvalid && wb + 8 < ngr) {
                                sc_nxt = __ldg(reinterpret_cast<const uint4*>(srow + wb + 8));
                                bc_nxt = __ldg(reinterpret_cast<const uint4*>(brow + wb + 8));
                            }
                        }
                        // both groups lie in the current window: windows start at multiples
                        // of 8 groups and a split pair is (2m, 2m + 1) for 32-input groups.
                        // The next window (still in flight) is only read at the slide above.
                        const int ia = ga - wb, ib = gb - wb;
                        sa = pick16(sc_cur, ia);
                        ba = pick16(bc_cur, ia);
                        sb = pick16(sc_cur, ib);
                        bb = pick16(bc_cur, ib);
                    } else if (rvalid) {
                        sa = __ldg(srow + ga);
                        ba = __ldg(brow + ga);
                        sb = __ldg(srow + gb);
                        bb = __ldg(brow + gb);
                    }
                    // this row's codes of k-block kb: k-block j starts at byte 8 * QB * j of
                    // the 128-byte swizzled row segment, chunk c at byte QB * c of the k-block
                    uint32_t words[kWordsPT * kWPC];
#pragma unroll
                    for (int v = 0; v < kPieces; ++v) {
                        const int c16 = j * QB / 2 + wd0 * QB / 16 + v;
                        const uint4 q4 = *reinterpret_cast<const uint4*>(rrow + ((c16 ^ (r & 7)) << 4));
                        words[4 * v] = q4.x; words[4 * v + 1] = q4.y;
                        words[4 * v + 2] = q4.z; words[4 * v + 3] = q4.w;
                    }
                    if (j == C::kRawKB - 1 || kb + 1 == ti.kb1) {
                        // the slot goes back to the code producer after its last k-block
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&rawempty[rs]);
                        if (++rs == C::kRawRing) { rs = 0; rph ^= 1u; }
                    }
                    // dequantise into registers first, so the math overlaps the wait for the
                    // operand slot (free once the MMA has consumed its previous contents)
                    uint4 dq8[kWordsPT];
                    const float sfa = __half2float(__ushort_as_half(sa));
                    const float bfa = __half2float(__ushort_as_half(ba));
                    if constexpr (QG != 32) {  // one group for all of this thread's chunks
                        const uint32_t s2 = pack_bf16x2(sfa, sfa), b2 = pack_bf16x2(bfa, bfa);
#pragma unroll
                        for (int w = 0; w < kWordsPT; ++w)
                            dq8[w] = QB == 4 ? dequant8(words[w], s2, b2)
                                             : dequant8_u8(words[2 * w], words[2 * w + 1], sfa, bfa);
                    } else {  // 32-input groups: chunk c of a k-block is in its group c / 4
                        const float sfb = __half2float(__ushort_as_half(sb));
                        const float bfb = __half2float(__ushort_as_half(bb));
#pragma unroll
                        for (int w = 0; w < kWordsPT; ++w) {
                            const bool second = ((wd0 + w) >> 2) != (wd0 >> 2);
                            const float sf = second ? sfb : sfa, bf = second ? bfb : bfa;
                            dq8[w] = QB == 4 ? dequant8(words[w], pack_bf16x2(sf, sf),
                                                        pack_bf16x2(bf, bf))
                                             : dequant8_u8(words[2 * w], words[2 * w + 1], sf, bf);
                        }
                    }
                    if (!mbar_wait(&empty[s], ph ^ 1u, abort)) { record_timeout(abort); ok = false; break; }
                    if constexpr (C::kTA) {
                        // weights -> this stage's TMEM columns of the warp's lane quarter
                        tc_fence_after();
                        const uint32_t tcol = tcol0 + (uint32_t)(s * C::kAStageCols);
#pragma unroll
                        for (int h = 0; h < kWordsPT / 4; ++h) {
                            uint32_t v16[16];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v16[4 * i] = dq8[4 * h + i].x; v16[4 * i + 1] = dq8[4 * h + i].y;
                                v16[4 * i + 2] = dq8[4 * h + i].z; v16[4 * i + 3] = dq8[4 * h + i].w;
                            }
                            tmem_st16(tcol + (uint32_t)(16 * h), v16);
                        }
                        tmem_st_wait();
                        tc_fence_before();
                    } else {
                        uint8_t* wrow_s = smem + s * C::kStageBytes + C::kXBytes + r * 128;
#pragma unroll
                        for (int w = 0; w < kWordsPT; ++w) {
                            const int c = wd0 + w;  // 16-byte chunk = 8 elements of the row
                            *reinterpret_cast<uint4*>(wrow_s + ((c ^ (r & 7)) << 4)) = dq8[w];
                        }
                        fence_proxy_async_smem();
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&full[s]);
                    if (++s == C::kStages) { s = 0; ph ^= 1u; }
                }
            }
        }
    } else {
        // ================================= epilogue =================================
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        int lt = 0;
        for (int t = tstart; t < total; t += tstep, ++lt) {
            const TileInfo ti = decode_tile<C>(p, prefix, rowoff, ngroups, t, crank);
            const int ab = C::kAccBufs == 2 ? (lt & 1) : 0;
            const uint32_t aph = (uint32_t)(C::kAccBufs == 2 ? (lt >> 1) : lt) & 1u;
            if (!mbar_wait(&tfull[ab], aph, abort)) { record_timeout(abort); break; }
            tc_fence_after();
            const uint32_t tacc0 =
                tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * C::kAccCols);
            if (!C::kSwap)
#pragma unroll 1
            for (int sub = 0; sub < C::kSub && sub * 128 < ti.rows; ++sub) {
                // accumulator row = token row (sub*128 + q*32 + lane), columns = features
                const uint32_t tacc = tacc0 + (uint32_t)(sub * 256);
                const int r = sub * 128 + q * 32 + lane;
                const bool valid = r < ti.rows;
                const long long orow = ti.out_row + r;
                if (MODE == kGateUp && C::kEpiBytes > 0) {
                    // h = silu(g) * u, kStgCols columns per staged chunk (see staged_store)
                    uint8_t* stg = smem + C::kEpiOff + q * (32 * C::kStgCols * 2);
                    const long long row0 = ti.out_row + sub * 128 + q * 32;
                    const int fbase = ti.f * 128;
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += C::kStgCols) {
#pragma unroll 1
                        for (int hh = 0; hh < C::kStgCols / 32; ++hh) {
                            uint32_t g[32], u[32];
                            __syncwarp();
                            tmem_ld32(tacc + c0 + 32 * hh, g);
                            tmem_ld32(tacc + 128 + c0 + 32 * hh, u);
                            tmem_ld_wait();
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint32_t w4[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int c = v * 8 + i * 2;
                                    w4[i] = pack_bf16x2(
                                        silu(__uint_as_float(g[c])) * __uint_as_float(u[c]),
                                        silu(__uint_as_float(g[c + 1])) * __uint_as_float(u[c + 1]));
                                }
                                stage_put<C::kStgCols>(stg, lane, 4 * hh + v,
                                                       make_uint4(w4[0], w4[1], w4[2], w4[3]));
                            }
                        }
                        __syncwarp();
                        staged_store<C::kStgCols>(stg, lane, static_cast<__nv_bfloat16_raw*>(p.out),
                                                  row0, p.out_ld, fbase + c0, sub * 128 + q * 32,
                                                  ti.rows, p.F);
                        __syncwarp();
                    }
                } else if (MODE == kGateUp) {
                    __nv_bfloat16_raw* dst = static_cast<__nv_bfloat16_raw*>(p.out) +
                                             orow * p.out_ld + (long long)ti.f * 128;
#pragma unroll 1
                    for (int c0 = 0; c0 < 128; c0 += 32) {
                        uint32_t g[32], u[32];
                        __syncwarp();
                        tmem_ld32(tacc + c0, g);
                        tmem_ld32(tacc + 128 + c0, u);
                        tmem_ld_wait();
                        if (valid) {
                            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
                            for (int v = 0; v < 4; ++v) {
                                uint32_t w4[4];
#pragma unroll
                                for (int i = 0; i < 4; ++i) {
                                    const int c = v * 8 + i * 2;
                                    w4[i] = pack_bf16x2(
                                        silu(__uint_as_float(g[c])) * __uint_as_float(u[c]),
                                        silu(__uint_as_float(g[c + 1])) * __uint_as_float(u[c + 1]));
                                }
                                d4[v] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                    }
                } else if (MODE == kDown && C::kEpiBytes > 0) {
                    uint8_t* stg = smem + C::kEpiOff + q * (32 * C::kStgCols * 2);
                    const int fbase = ti.f * 256;
                    const long long row0 = ti.out_row + sub * 128 + q * 32;
#pragma unroll 1
                    for (int c0 = 0; c0 < 256 && fbase + c0 < p.F; c0 += C::kStgCols) {
#pragma unroll 1
                        for (int hh = 0; hh < C::kStgCols / 32; ++hh) {
                            uint32_t a[32];
                            __syncwarp();
                            tmem_ld32(tacc + c0 + 32 * hh, a);
                            tmem_ld_wait();
#pragma unroll
                            for (int v = 0; v < 4; ++v)
                                stage_put<C::kStgCols>(
                                    stg, lane, 4 * hh + v,
                                    make_uint4(pack_bf16x2(__uint_as_float(a[8 * v + 0]), __uint_as_float(a[8 * v + 1])),
                                               pack_bf16x2(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                                               pack_bf16x2(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                                               pack_bf16x2(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7]))));
                        }
                        __syncwarp();
                        staged_store<C::kStgCols>(stg, lane, static_cast<__nv_bfloat16_raw*>(p.out),
                                                  row0, p.out_ld, fbase + c0, sub * 128 + q * 32,
                                                  ti.rows, p.F);
                        __syncwarp();
                    }
                } else {
                    const int fbase = ti.f * 256;
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 32) {
                        uint32_t a[32];
                        __syncwarp();
                        tmem_ld32(tacc + c0, a);
                        tmem_ld_wait();
                        if (valid && fbase + c0 < p.F) {
                        if (MODE == kDown) {
                            __nv_bfloat16_raw* dst = static_cast<__nv_bfloat16_raw*>(p.out) +
                                                     orow * p.out_ld + fbase + c0;
                            if (fbase + c0 + 32 <= p.F) {
                                uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
                                for (int v = 0; v < 4; ++v)
                                    d4[v] = make_uint4(
                                        pack_bf16x2(__uint_as_float(a[v * 8 + 0]), __uint_as_float(a[v * 8 + 1])),
                                        pack_bf16x2(__uint_as_float(a[v * 8 + 2]), __uint_as_float(a[v * 8 + 3])),
                                        pack_bf16x2(__uint_as_float(a[v * 8 + 4]), __uint_as_float(a[v * 8 + 5])),
                                        pack_bf16x2(__uint_as_float(a[v * 8 + 6]), __uint_as_float(a[v * 8 + 7])));
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (fbase + c0 + i < p.F)
                                        dst[i].x = (unsigned short)(pack_bf16x2(__uint_as_float(a[i]), 0.0f) & 0xFFFFu);
                            }
                        } else {
                            float* dst = static_cast<float*>(p.out) + (long long)ti.ks * p.split_stride +
                                         orow * p.out_ld + fbase + c0;
                            if (fbase + c0 + 32 <= p.F && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
                                // whole 16-byte pieces of the row (the scalar form cost the
                                // prefill router most of its time)
                                float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
                                for (int v = 0; v < 8; ++v)
                                    d4[v] = make_float4(__uint_as_float(a[4 * v]), __uint_as_float(a[4 * v + 1]),
                                                        __uint_as_float(a[4 * v + 2]), __uint_as_float(a[4 * v + 3]));
                            } else {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    if (fbase + c0 + i < p.F) dst[i] = __uint_as_float(a[i]);
                            }
                        }
                        }
                    }
                }
            } else {
                // accumulator row = feature (q*32 + lane), columns = tokens
                const uint32_t tacc = tacc0;
                const int feat = ti.f * 128 + q * 32 + lane;
                const bool fvalid = feat < p.F;
#pragma unroll 1
                for (int j0 = 0; j0 < C::kTok; j0 += 16) {
                    uint32_t a[16], b[16];
                    __syncwarp();
                    tmem_ld16(tacc + j0, a);
                    if (MODE == kGateUp) tmem_ld16(tacc + C::kTok + j0, b);
                    tmem_ld_wait();
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = j0 + jj;
                        if (!fvalid || j >= ti.rows) break;
                        const long long orow = ti.out_row + j;
                        if (MODE == kGateUp) {
                            const float h = silu(__uint_as_float(a[jj])) * __uint_as_float(b[jj]);
                            static_cast<__nv_bfloat16_raw*>(p.out)[orow * p.out_ld + feat].x =
                                (unsigned short)(pack_bf16x2(h, 0.0f) & 0xFFFFu);
                        } else if (MODE == kDown) {
                            static_cast<__nv_bfloat16_raw*>(p.out)[orow * p.out_ld + feat].x =
                                (unsigned short)(pack_bf16x2(__uint_as_float(a[jj]), 0.0f) & 0xFFFFu);
                        } else {
                            static_cast<float*>(p.out)[(long long)ti.ks * p.split_stride +
                                                       orow * p.out_ld + feat] = __uint_as_float(a[jj]);
                        }
                    }
                }
            }
            tc_fence_before();
            if constexpr (C::kPair) {
                // one arrival per warp, on the leader's barrier (remote for the peer)
                __syncwarp();
                if (lane == 0) {
                    if (leader) mbar_arrive(&tempty[ab]);
                    else mbar_arrive_cluster(&tempty[ab], 0);
                }
            } else {
                mbar_arrive(&tempty[ab]);
            }
        }
    }

    // ---- tear-down ----
    // the next kernel may start launching now (not earlier: its blocks would sit resident
    // through this kernel's whole main loop)
    pdl_launch_dependents();
    tc_fence_before();
    __syncthreads();
    // a pair: neither CTA leaves while the other's UMMAs, copies or arrivals may still touch
    // its shared memory or TMEM
    if constexpr (C::kPair) cluster_sync();
    if (warp == 1) {
        tc_fence_after();
        if constexpr (C::kPair) tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

// ------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] (cols contiguous), box of 64 columns x box_rows rows,
// 128-byte swizzle, out-of-range elements read as zero.
bool make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    if (rows < 1) rows = 1;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D uint32 tensor [rows, cols_u32] of packed codes, box of 32 words (one 128-byte row
// segment: 256 4-bit or 128 8-bit codes) x box_rows rows, 128-byte swizzle.
bool make_map_q4(CUtensorMap* m, const void* base, long long rows, long long cols_u32,
                 int box_rows) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    if (rows < 1) rows = 1;
    const cuuint64_t dims[2] = {(cuuint64_t)cols_u32, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols_u32 * 4};
    const cuuint32_t box[2] = {32u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int TOKT, int QB, int QG, int PAIR = 0>
cudaError_t run_gemm(const GemmArgs& a, cudaStream_t s) {
    using C = Cfg<MODE, TOKT, QB, PAIR>;
    constexpr bool Q4 = C::kQ;
    static DeviceOnce attr_once;
    const cudaError_t attr_err = attr_once.run([] {
        return cudaFuncSetAttribute(moe_gemm_kernel<MODE, TOKT, QB, QG, PAIR>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    });
    if (attr_err != cudaSuccess) return attr_err;

    const int wbox = C::kSwap ? 128 : (C::kPair || MODE == kGateUp ? 128 : 256);
    const long long wrows_routed = (long long)(a.offsets ? a.E : 1) * a.F;
    CUtensorMap m_act, m_act_sh, m_w0, m_w1, m_sw0, m_sw1;
    bool ok = make_map(&m_act, a.act, a.act_rows, a.Kdim, C::kTok);
    ok = ok && make_map(&m_act_sh, a.act_shared ? a.act_shared : a.act,
                        a.act_shared ? (a.shared_act_row0 + a.shared_rows) : a.act_rows, a.Kdim,
                        C::kTok);
    if (Q4) {
        const long long words = (long long)a.Kdim * QB / 32;  // uint32 words of codes per row
        ok = ok && make_map_q4(&m_w0, a.w.w0, wrows_routed, words, wbox);
        ok = ok && make_map_q4(&m_w1, a.w.w1 ? a.w.w1 : a.w.w0, wrows_routed, words, wbox);
    } else {
        ok = ok && make_map(&m_w0, a.w.w0, wrows_routed, a.Kdim, wbox);
        ok = ok && make_map(&m_w1, a.w.w1 ? a.w.w1 : a.w.w0, wrows_routed, a.Kdim, wbox);
    }
    // shared expert maps are bf16 (a stand-in view of the act tensor when there is none)
    const void* sw0 = a.has_shared ? a.ws.w0 : a.act;
    const void* sw1 = a.has_shared ? (a.ws.w1 ? a.ws.w1 : a.ws.w0) : a.act;
    const long long srows = a.has_shared ? a.F : a.act_rows;
    ok = ok && make_map(&m_sw0, sw0, srows, a.Kdim, wbox);
    ok = ok && make_map(&m_sw1, sw1, srows, a.Kdim, wbox);
    if (!ok) return cudaErrorInvalidValue;

    KParams p;
    p.offsets = a.offsets;
    p.single_rows = a.single_rows;
    p.E = a.E;
    p.has_shared = a.has_shared;
    p.shared_rows = a.shared_rows;
    p.shared_act_row0 = a.shared_act_row0;
    p.shared_out_row0 = a.shared_out_row0;
    p.Kdim = a.Kdim;
    p.F = a.F;
    p.ksplit = a.ksplit;
    p.split_stride = a.split_stride;
    p.out = a.out;
    p.out_ld = a.out_ld;
    p.qscale[0] = static_cast<const unsigned short*>(a.w.s0);
    p.qbias[0] = static_cast<const unsigned short*>(a.w.b0);
    p.qscale[1] = static_cast<const unsigned short*>(a.w.s1);
    p.qbias[1] = static_cast<const unsigned short*>(a.w.b1);
    auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    p.qgroup = Q4 ? a.w.group : kBK;
    p.q_vec = Q4 && (a.Kdim / p.qgroup) % 8 == 0 && al16(a.w.s0) && al16(a.w.b0) &&
              (MODE != kGateUp || (al16(a.w.s1) && al16(a.w.b1)));

    long long grid = num_sms();
    if (a.max_tiles < grid) grid = a.max_tiles;
    if (grid < 1) return cudaSuccess;
    if constexpr (C::kPair) {
        // persistent CTA pairs: clusters of two, one CTA per SM, as many pairs as the device
        // can hold at once (an SM left over in a GPC of odd size takes no pair)
        cudaLaunchConfig_t cfg = {};
        cfg.blockDim = dim3(C::kThreadsCta, 1, 1);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        static int resident[DeviceOnce::kMaxDevices] = {};
        static DeviceOnce occ_once;
        int dev = 0;
        cudaError_t err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        if (dev < 0 || dev >= DeviceOnce::kMaxDevices) return cudaErrorInvalidDevice;
        err = occ_once.run([&] {
            cfg.gridDim = dim3((unsigned)(2 * (num_sms() / 2)), 1, 1);
            int n = 0;
            const cudaError_t e = cudaOccupancyMaxActiveClusters(
                &n, moe_gemm_kernel<MODE, TOKT, QB, QG, PAIR>, &cfg);
            if (e == cudaSuccess) resident[dev] = n > 0 ? n : 1;
            return e;
        });
        if (err != cudaSuccess) return err;
        long long pairs = resident[dev];
        if (num_sms() / 2 < pairs) pairs = num_sms() / 2;
        if (a.max_tiles < pairs) pairs = a.max_tiles;
        if (pairs < 1) pairs = 1;
        cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
        cfg.numAttrs = pdl_enabled() ? 2 : 1;
        err = cudaLaunchKernelEx(&cfg, moe_gemm_kernel<MODE, TOKT, QB, QG, PAIR>,
                                                   m_act, m_act_sh, m_w0, m_w1, m_sw0, m_sw1, p);
        return err != cudaSuccess ? err : cudaGetLastError();
    }
    return launch_kernel(moe_gemm_kernel<MODE, TOKT, QB, QG, PAIR>, dim3((unsigned)grid),
                         dim3(C::kThreadsCta), (size_t)C::kSmemBytes, s, m_act, m_act_sh, m_w0,
                         m_w1, m_sw0, m_sw1, p);
}

// Token tiles: the router takes 16 / 32 / 64 / 128 tokens on N or 128 on M; the expert
// GEMMs take 64 / 128 tokens on N or 128 on M (128 on N bf16 only: the quantised TMEM-A path
// has no TMEM room for it).
template <int MODE, int QB, int QG>
cudaError_t dispatch_tok(const GemmArgs& a, cudaStream_t s) {
    switch (a.tok_tile) {
        case 0:
            if constexpr (QB == 0 && MODE != kRouter)
                if (a.pair) return run_gemm<MODE, 0, QB, QG, 1>(a, s);
            return run_gemm<MODE, 0, QB, QG>(a, s);
        case 16:
            if constexpr (MODE == kRouter) return run_gemm<MODE, 16, QB, QG>(a, s);
            return cudaErrorInvalidValue;
        case 32:
            if constexpr (MODE == kRouter) return run_gemm<MODE, 32, QB, QG>(a, s);
            return cudaErrorInvalidValue;
        case 64: return run_gemm<MODE, 64, QB, QG>(a, s);
        case 128:
            if constexpr (QB == 0) return run_gemm<MODE, 128, QB, QG>(a, s);
            return cudaErrorInvalidValue;
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t s) {
    if (a.w.bits == 4 || a.w.bits == 8) {
        if (a.ws.bits != 16 && a.has_shared) return cudaErrorInvalidValue;
        if (a.w.group != 32 && a.w.group != 64 && a.w.group != 128) return cudaErrorInvalidValue;
        if (a.mode == kRouter) return cudaErrorInvalidValue;  // the router is always bf16
        const bool gu = a.mode == kGateUp;
#define MOE_Q_DISPATCH(QB, QG) \
    return gu ? dispatch_tok<kGateUp, QB, QG>(a, s) : dispatch_tok<kDown, QB, QG>(a, s)
        if (a.w.bits == 4) {
            if (a.w.group == 32) MOE_Q_DISPATCH(4, 32);
            if (a.w.group == 128) MOE_Q_DISPATCH(4, 128);
            MOE_Q_DISPATCH(4, 64);
        }
        if (a.w.group == 32) MOE_Q_DISPATCH(8, 32);
        if (a.w.group == 128) MOE_Q_DISPATCH(8, 128);
        MOE_Q_DISPATCH(8, 64);
#undef MOE_Q_DISPATCH
    }
    if (a.w.bits != 16) return cudaErrorInvalidValue;
    switch (a.mode) {
        case kGateUp: return dispatch_tok<kGateUp, 0, 0>(a, s);
        case kDown: return dispatch_tok<kDown, 0, 0>(a, s);
        case kRouter: return dispatch_tok<kRouter, 0, 0>(a, s);
    }
    return cudaErrorInvalidValue;
}

namespace {
// A single warp: lane 0 initialises an mbarrier expecting one arrival that never comes and
// waits on it through mbar_wait with the given limit, exactly as a GEMM role waits on a
// copy that never lands; when the wait gives up it records the timeout.
__global__ void watchdog_selftest_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, &abort_flag, limit_ns))
        record_timeout(&abort_flag);
}
}  // namespace

cudaError_t launch_watchdog_selftest(unsigned long long limit_ns, cudaStream_t s) {
    watchdog_selftest_kernel<<<1, 32, 0, s>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t read_device_status(unsigned int* out, int clear, cudaStream_t s) {
    cudaError_t err = cudaMemcpyFromSymbolAsync(out, g_status, sizeof(unsigned int), 0,
                                                cudaMemcpyDeviceToHost, s);
    if (err != cudaSuccess) return err;
    err = cudaStreamSynchronize(s);
    if (err != cudaSuccess || !clear) return err;
    const unsigned int zero = 0;
    err = cudaMemcpyToSymbolAsync(g_status, &zero, sizeof(unsigned int), 0,
                                  cudaMemcpyHostToDevice, s);
    if (err != cudaSuccess) return err;
    return cudaStreamSynchronize(s);
}

int num_sms() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return n > 0 ? n : 1;
}

}  // namespace moe
