// gemm.cu -- W4A4 block-scaled FP4 GEMM on the 5th-generation tensor cores.
//
//   out[m, n] = bf16_rne( sum_k A[m, k] * B[n, k] + bias[n] )
//
// Both operands are MXFP4 ("Efficiently Serving NVFP4 Models on AMD
// Instinct MI350X/MI355X ... via Online NVFP4 to Quark MXFP4
// Requantization", "Native FP4 matmul": dense layers and MoE experts run on
// native block-scaled FP4 matrix instructions with no separate dequantize
// step); the bf16 output with a bf16 per-output-channel bias follows "W4A4
// MXFP4 Quantization" (Configuration) and "[SGLang] FP4 ..." (section 6).
//
// Design: one persistent CTA per SM walks output tiles (the MMA-M operand's
// 128-row tile fastest).  A pipeline stage holds KC slabs of 128 packed
// bytes (256 elements) of K for both operands.  12 to 16 warps (the
// register-split configurations below add two idle warps):
//   warp 0      TMA producer: per (tile, stage) one tensor-map load per
//               operand (a 3-D box spanning the KC slabs when KC > 1: the
//               TMA unit keeps only a few copies in flight per SM, so fewer,
//               larger copies stream faster) plus one bulk copy of the
//               matching scale chunks per 128-row scale tile, into a ring of
//               smem stages that runs on across tile boundaries.
//   warp 1      TMEM owner and MMA issuer: per stage, 4 * KC tcgen05.mma
//               kind::mxf4 (K = 64, two E8M0 scales per row each) accumulate
//               into a 128 x BN fp32 TMEM tile; tcgen05.commit frees the
//               stage, and at the end of a tile signals the epilogue.  This
//               thread's own instructions pace the narrow decode MMAs (a
//               barrier wait costs it a few hundred cycles even when the
//               phase is complete), so it waits once per stage, on the scale
//               movers' barrier (they copy only after the stage has landed),
//               and forms descriptors from precomputed bases.
//   CPW warps   scale movers (warps 2 .. 1+CPW; 4, or 2 where the epilogue
//               needs the registers): per stage, tcgen05.cp of the scale
//               chunks from smem into that stage's TMEM scale columns, split
//               between the warps.  A thread's copies run one after another at about
//               a hundred cycles each, so one thread issuing both copies and
//               MMAs would serialise them; on separate threads they overlap
//               the MMAs of the previous stage.
//   8 warps     epilogue (the last eight): each warp reads 32 TMEM lanes x BN/2 columns into
//               registers, releases the accumulator at once (so the next
//               tile's MMAs start), adds bias, rounds to bf16, stages its
//               part of the tile in its own shared-memory area and writes it
//               with TMA tensor stores.
// Orientation: the MMA-M operand is A (activations) in the normal mode and
// the weights in the swapped mode used for small M (decode); there the
// tokens are the MMA N dimension and the staged tile is the transpose.
// Split-K (swapped mode, at most half the SMs busy otherwise, caller
// workspace): the tiles' K stages form one sequence of units cut into equal
// contiguous ranges, one per CTA, with S CTAs per tile so that a range never
// leaves its tile.  The CTA holding a tile's first K stages finishes it: it
// adds the fp32 partial sums the other S - 1 CTAs left in the workspace, in
// K order (a fixed reduction order, so results do not vary from run to run),
// then runs the epilogue.  Such a launch is cooperative (its CTAs wait on
// one another).
// Operand formats (kFmt):
//   kFmtMx  both operands MXFP4 (the path above);
//   kFmtNv  both operands NVFP4 as "[SGLang] FP4 ..." sections 5-6
// run them on hardware with native NVFP4: one E4M3 scale per 16 elements
// (two 512-byte scale chunks per 128 elements of K instead of one, four
// scales per row per K = 64 step, tcgen05.mma kind::mxf4nvf4 with
// scale_vec::4X) and a per-tensor alpha applied to the accumulator in the
// epilogue before the bias;
//   kFmtA8  the W4A8 fallback of "W4A4 MXFP4 Quantization" (MXFP8
// activations with the same MXFP4 weights): E4M3 activations (one byte per
// element) and the FP4 weights, which TMA expands to one element per byte
// in shared memory (16 codes in the low half of every 16 bytes), so both
// operands stage 128 elements of K per 128-byte row; tcgen05.mma
// kind::mxf8f6f4 (K = 32, one E8M0 scale per row each, chosen by the
// descriptor's byte selector).
// Every mbarrier wait is bounded; on expiry the kernel records a timeout in
// the status word and winds down.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace fp4lin {

namespace {

constexpr int BM = 128;
constexpr int kSlabBytes = 128;  // packed bytes of K per row per slab (256 elements)
constexpr int kEpiWarps = 8;

enum : int { kFmtMx = kGemmMx, kFmtNv = kGemmNv, kFmtA8 = kGemmW4A8, kFmtDual = kGemmDual };

struct GemmParams {
    int64_t units;              // split-K: total K-stage units (0: one CTA per whole tile)
    uint32_t* flags;            // split-K: per-CTA partial-ready counters (zero between calls)
    float* partials;            // split-K: per-CTA partial tile [BN][128] fp32
    const uint8_t* sfa;         // swizzled scales of the MMA-M operand
    const uint8_t* sfb;         // swizzled scales of the MMA-N operand (per expert when grouped)
    const __nv_bfloat16* bias;  // per output channel (per expert when grouped)
    __nv_bfloat16* out;
    const int32_t* offsets;     // grouped: row offsets [E+1]
    int E;
    int rows_a;                 // rows of the MMA-M operand (normal: M, swapped: N)
    int rows_b;                 // rows of the MMA-N operand per expert (normal: N, swapped: M)
    int K;
    int kb4;                    // K / 128: scale-factor column groups per row tile
    int m_tiles;                // MMA-M tiles (grouped: bound on sum_e ceil(rows_e / 128))
    int n_tiles;
    int ldo;                    // output row stride (elements) = the problem's N
    int64_t sfb_expert_stride;
    float alpha;                // NVFP4 mode: factor on the accumulator before the bias
    int early_w;                // weights not written by the kernel this one may overlap
    int withhold_signal;        // test hook: the last CTA of a split launch never publishes its partial
    const uint16_t* x;          // fused activation quantization: bf16 tokens [rows_b, K] (swapped mode)
    const uint16_t* xmul;       // its smooth pre-scale (bf16 [K]) or null
    int x_uos;                  // its block rule: UOS (else OCP)
    const float* coarse;        // DualScale: coarse weight scales [weight rows][K / 512]
    unsigned long long wait_ns; // limit of every bounded wait
    unsigned int* status;
};

template <int BN, int STAGES, int KC, int CPW, bool kSwap, int kFmt>
struct Cfg {
    static constexpr bool kNv = kFmt == kFmtNv;
    static constexpr bool kA8 = kFmt == kFmtA8;
    // DualScale: a stage is one 512-element coarse group of K, and its MMAs
    // write one of two TMEM partial buffers in turn
    static constexpr bool kDual = kFmt == kFmtDual;
    static_assert(!kDual || KC == 2, "DualScale: one 512-element group per stage");
    // Four scale warps beside a 256-wide epilogue do not fit the register
    // file at 14 warps: 16 warps then, warps 6-7 idle, and the two non-
    // epilogue warpgroups hand registers to the epilogue ones (setmaxnreg).
    static constexpr bool SPLIT = BN == 256 && CPW > 2;
    static constexpr int REGS_LOW = 80;    // warps 0-7 after the split
    static constexpr int REGS_HIGH = 176;  // epilogue warps after the split
    // the two halves of the split fill the 65536 registers of 16 warps x 32 x 128
    static_assert(!SPLIT || (REGS_LOW + REGS_HIGH) * 256 == 65536, "register split must fill the register file");
    static constexpr int FIRST_EPI_WARP = SPLIT ? 8 : 2 + CPW;
    static constexpr int THREADS = 32 * (FIRST_EPI_WARP + kEpiWarps);
    // a slab is one 128-byte row per operand row: 256 elements of K (packed
    // FP4) or 128 (W4A8: E4M3, and FP4 expanded to a byte per element)
    static constexpr int GROUPS = kA8 ? KC : 2 * KC;  // 128-element groups of K per stage
    static constexpr int MMAS_PER_GROUP = kA8 ? 4 : 2;  // K = 32 (W4A8) or 64 per MMA
    static constexpr int APG = kNv ? 2 : 1;  // 512-byte scale chunks per group and 128-row tile
    static constexpr int ATOMS = GROUPS * APG;  // scale chunks per stage and 128-row tile
    static constexpr int A_BYTES = BM * kSlabBytes * KC;  // shared memory per stage
    static constexpr int B_BYTES = BN * kSlabBytes * KC;
    // bytes the TMA counts per stage: the expanded FP4 operand (the weights:
    // MMA-M side when swapped) counts its global bytes, half its footprint
    static constexpr int A_TX = (kA8 && kSwap) ? A_BYTES / 2 : A_BYTES;
    static constexpr int B_TX = (kA8 && !kSwap) ? B_BYTES / 2 : B_BYTES;
    static constexpr int SFB_TILES = (BN + 127) / 128;
    static constexpr int SFA_BYTES = ATOMS * 512;
    static constexpr int SFB_BYTES = SFB_TILES * ATOMS * 512;
    // normal-mode store chunk: 32 rows x CHUNK columns per warp (16 where the
    // NVFP4 scale chunks need the shared memory for a fourth stage)
    static constexpr int CHUNK = (kNv && BN == 256) ? 16 : 32;
    static constexpr int EPI_WARP_BYTES = kSwap ? 32 * (BN / 2) * 2 : 32 * CHUNK * 2;
    static constexpr int EPI_BYTES = kEpiWarps * EPI_WARP_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_SFA = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_SFB = OFF_SFA + STAGES * SFA_BYTES;
    static constexpr int OFF_EPI = OFF_SFB + STAGES * SFB_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + EPI_BYTES;
    static constexpr int NUM_BARS = 3 * STAGES + 2 + (kDual ? 4 : 0);
    static constexpr int OFF_TMEM_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_PREFIX = OFF_TMEM_SLOT + 16;
    static constexpr int SMEM_FIXED = OFF_PREFIX + 1024;  // + 1 KB alignment slack
    static constexpr int SF_COLS_A = 4 * ATOMS;
    static constexpr int SF_COLS_B_ATOM = 4 * SFB_TILES;
    static constexpr int SF_COLS = SF_COLS_A + ATOMS * SF_COLS_B_ATOM;
    static constexpr int TMEM_USED = (kDual ? 2 : 1) * BN + STAGES * SF_COLS;  // one scale buffer per smem stage
    static constexpr int TMEM_COLS = TMEM_USED <= 32 ? 32 : TMEM_USED <= 64 ? 64 : TMEM_USED <= 128 ? 128
                                     : TMEM_USED <= 256 ? 256 : 512;
    static_assert(TMEM_USED <= 512, "TMEM overflow");
    static_assert(OFF_EPI % 1024 == 0, "staging alignment (swizzled store boxes)");
    static_assert(SMEM_FIXED <= 232448, "shared memory budget");
    static constexpr int CW = BN / 2;  // accumulator columns per epilogue warp
    static_assert(kSwap || CW % CHUNK == 0, "normal-mode columns per warp must be whole store chunks");
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

struct Tile {
    int64_t a_row0;  // first MMA-M row
    int rows_valid;  // MMA-M rows of this tile inside the problem (inside the expert when grouped)
    int sfa_rt;      // scale row tile of the MMA-M operand
    int n0;          // first MMA-N row
    int expert;
    bool valid;
};

template <int BN, bool kGrouped>
__device__ __forceinline__ Tile decode_tile(int t, const GemmParams& p, const int32_t* tiles_before)
{
    Tile T;
    T.expert = 0;
    T.valid = true;
    int rows;
    if constexpr (kGrouped) {
        // expert-major walk: all tiles of expert e (its 128-row tiles fastest,
        // then its weight tiles) before those of e + 1, so the CTAs running
        // at once share a few experts' weights and activations in L2
        const int nt = p.n_tiles;
        if (t >= tiles_before[p.E] * nt) {
            T.valid = false;
            T.rows_valid = 0;
            return T;
        }
        int lo = 0, hi = p.E;  // tiles_before[lo] * nt <= t < tiles_before[hi] * nt
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tiles_before[mid] * nt <= t)
                lo = mid;
            else
                hi = mid;
        }
        const int mt = tiles_before[lo + 1] - tiles_before[lo];  // >= 1: expert lo holds tile t
        const int local = t - tiles_before[lo] * nt;
        const int gl = local % mt;
        int start, rows_e;
        group_rows(p.offsets, lo, p.rows_a, &start, &rows_e);
        T.expert = lo;
        T.n0 = (local / mt) * BN;
        T.sfa_rt = min(tiles_before[lo] + gl, p.m_tiles - 1);  // inside the scale array whatever the offsets
        T.a_row0 = start + static_cast<int64_t>(gl) * BM;
        rows = rows_e - gl * BM;
    } else {
        const int g = t % p.m_tiles;
        T.n0 = (t / p.m_tiles) * BN;
        T.sfa_rt = g;
        T.a_row0 = static_cast<int64_t>(g) * BM;
        rows = p.rows_a - g * BM;
    }
    T.rows_valid = rows < BM ? rows : BM;
    return T;
}

template <int CW>
__device__ __forceinline__ void tmem_load_cols(uint32_t taddr, uint32_t* v)
{
    if constexpr (CW == 8) {
        tmem_ld_32x32b_x8(taddr, v);
    } else if constexpr (CW == 16) {
        tmem_ld_32x32b_x16(taddr, v);
    } else {
#pragma unroll
        for (int c = 0; c < CW; c += 32)
            tmem_ld_32x32b_x32(taddr + c, v + c);
    }
}

// A CTA's work: whole tiles t = blockIdx.x, + gridDim.x, ... or, in split-K
// mode, the segments of its unit range [u0, u1) (unit = tile * nkb + stage).
enum WorkMode { kWhole = 0, kHead = 1, kPartial = 2 };

struct Work {
    int t;
    int kb0, kb1;  // stages [kb0, kb1) of tile t
    int mode;      // kWhole; kHead: first stages, adds the others' partials; kPartial: later stages
};

struct WorkIter {
    int64_t cur, end;
    bool split;
};

__device__ __forceinline__ WorkIter work_begin(const GemmParams& p, int total_tiles)
{
    WorkIter w;
    w.split = p.units > 0;
    if (w.split) {
        w.cur = static_cast<int64_t>(blockIdx.x) * p.units / gridDim.x;
        w.end = static_cast<int64_t>(blockIdx.x + 1) * p.units / gridDim.x;
    } else {
        w.cur = blockIdx.x;
        w.end = total_tiles;
    }
    return w;
}

__device__ __forceinline__ bool work_next(WorkIter& it, int nkb, Work& w)
{
    if (it.cur >= it.end)
        return false;
    if (it.split) {
        w.t = static_cast<int>(it.cur / nkb);
        const int64_t base = static_cast<int64_t>(w.t) * nkb;
        w.kb0 = static_cast<int>(it.cur - base);
        w.kb1 = static_cast<int>(min(it.end - base, static_cast<int64_t>(nkb)));
        w.mode = w.kb0 > 0 ? kPartial : (w.kb1 < nkb ? kHead : kWhole);
        it.cur = base + w.kb1;
    } else {
        w.t = static_cast<int>(it.cur);
        w.kb0 = 0;
        w.kb1 = nkb;
        w.mode = kWhole;
        it.cur += gridDim.x;
    }
    return true;
}

// Split-K: the CTA whose unit range holds unit u.
__device__ __forceinline__ int unit_owner(int64_t u, int64_t units)
{
    return static_cast<int>(((u + 1) * gridDim.x - 1) / units);
}

// Release add at GPU scope: the warp's earlier writes (ordered before it by a
// __syncwarp) are visible to whoever acquires the counter afterwards.
__device__ __forceinline__ void red_release_add_gpu(uint32_t* p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <int KC>
__device__ __forceinline__ void load_operand(void* dst, const CUtensorMap* map, uint64_t* bar, int kb, int64_t row0)
{
    if constexpr (KC == 1)
        tma_load_2d(dst, map, bar, kb * kSlabBytes, static_cast<int32_t>(row0));
    else
        tma_load_3d(dst, map, bar, 0, static_cast<int32_t>(row0), kb * KC);
}

// kFuseX (swapped MXFP4 only): the tokens arrive as bf16 and the epilogue
// warps, idle during the main loop, quantize each stage's token slab into the
// stage's B operand and scale chunk themselves (the activation quantizer's
// block arithmetic, so the codes and scales are the same bytes), instead of
// a TMA load of tokens quantized by a kernel before this one.
template <int BN, int STAGES, int KC, int CPW, bool kSwap, bool kGrouped, int kFmt, bool kFuseX = false>
__global__ void __launch_bounds__(Cfg<BN, STAGES, KC, CPW, kSwap, kFmt>::THREADS, 1)
    gemm_fp4_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmO, const GemmParams p)
{
    using C = Cfg<BN, STAGES, KC, CPW, kSwap, kFmt>;
    constexpr bool kNv = C::kNv, kA8 = C::kA8;
    constexpr int kFirstEpiWarp = C::FIRST_EPI_WARP;
    static_assert(!kFuseX || (kSwap && !kGrouped && kFmt == kFmtMx && BN <= 128), "fused quantization: swapped MXFP4");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;
    uint64_t* sf_full = empty + STAGES;
    uint64_t* accum_full = sf_full + STAGES;
    uint64_t* accum_empty = accum_full + 1;
    uint64_t* part_full = accum_empty + 1;  // DualScale: partial buffer b holds a finished group
    uint64_t* part_empty = part_full + 2;   // DualScale: the epilogue has read partial buffer b
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
    int32_t* tiles_before = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int total_tiles = p.m_tiles * p.n_tiles;
    const int nkb = (p.kb4 + C::GROUPS - 1) / C::GROUPS;  // stages per tile

    // Loads of one stage (producer thread): the weight half (the MMA-M
    // operand when swapped, else the MMA-N one, with its scale chunks), the
    // activation half, or both; `expect` posts the whole stage's bytes.
    enum { kHalfW = 1, kHalfX = 2 };
    auto stage_loads = [&](int s, int kb, const Tile& T, int halves, bool expect) {
        const int64_t b_row0 = static_cast<int64_t>(T.expert) * p.rows_b + T.n0;
        const uint8_t* sfb = p.sfb + static_cast<int64_t>(T.expert) * p.sfb_expert_stride;
        int nsfb = (p.rows_b + 127) / 128 - T.n0 / 128;
        nsfb = nsfb < C::SFB_TILES ? nsfb : C::SFB_TILES;
        const int groups = min(C::GROUPS, p.kb4 - C::GROUPS * kb);
        const uint32_t sf_bytes = static_cast<uint32_t>(groups * C::APG) * 512u;
        const int64_t atoms_per_rt = static_cast<int64_t>(p.kb4) * C::APG;  // chunks per 128-row tile
        // boxes past the end of K or of the rows are zero-filled and still counted
        if (expect)
            mbar_arrive_expect_tx(&full[s], kFuseX ? C::A_TX + sf_bytes : C::A_TX + C::B_TX + sf_bytes * (1u + nsfb));
        const int a_half = kSwap ? kHalfW : kHalfX;
        if (halves & a_half) {
            load_operand<KC>(smem + C::OFF_A + s * C::A_BYTES, &tmA, &full[s], kb, T.a_row0);
            bulk_load(smem + C::OFF_SFA + s * C::SFA_BYTES, p.sfa + (T.sfa_rt * atoms_per_rt + C::ATOMS * kb) * 512,
                      sf_bytes, &full[s]);
        }
        if (halves & (kHalfW | kHalfX) & ~a_half) {
            load_operand<KC>(smem + C::OFF_B + s * C::B_BYTES, &tmB, &full[s], kb, b_row0);
            for (int j = 0; j < nsfb; ++j)
                bulk_load(smem + C::OFF_SFB + s * C::SFB_BYTES + j * C::ATOMS * 512,
                          sfb + ((T.n0 / 128 + j) * atoms_per_rt + C::ATOMS * kb) * 512, sf_bytes, &full[s]);
        }
    };

    // ------------------------------------------------------------ setup
    // (no global memory is touched before the dependency wait: this part
    // overlaps the previous kernel in the stream -- except, when the caller
    // states that the weights are not written by that kernel, the weight
    // half of the first stages of this CTA's first tile)
    int npre = 0;  // producer thread: stages whose weight half is already in flight
    // Producer thread: its first work item, decoded before the dependency
    // wait (a chain of dependent integer operations on the launch parameters,
    // ~0.5 us on one thread) so that it overlaps the previous kernel.
    WorkIter first_wi{};
    Work first_w{};
    Tile first_t{};
    bool have_first = false;
    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], kFuseX ? 1 + kEpiWarps : 1);  // fused: + one arrival per quantizing warp
            mbar_init(&empty[s], 1);
            mbar_init(&sf_full[s], CPW);
        }
        mbar_init(accum_full, 1);
        mbar_init(accum_empty, kEpiWarps);
        if constexpr (C::kDual) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(&part_full[b], 1);
                mbar_init(&part_empty[b], kEpiWarps);
            }
        }
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmO);
        if constexpr (!kGrouped) {
            first_wi = work_begin(p, total_tiles);
            have_first = work_next(first_wi, nkb, first_w);
            if (have_first) {
                first_t = decode_tile<BN, false>(first_w.t, p, nullptr);
                if (p.early_w) {
                    npre = min(STAGES, first_w.kb1 - first_w.kb0);
                    for (int i = 0; i < npre; ++i)
                        stage_loads(i, first_w.kb0 + i, first_t, kHalfW, true);
                }
            }
        }
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    grid_dependency_wait();
    launch_dependents();
    if constexpr (kGrouped) {
        if (warp == 2) {
            // exclusive prefix of per-expert 128-row tile counts
            int carry = 0;
            for (int base = 0; base <= p.E; base += 32) {
                const int e = base + lane;
                int t = 0;
                if (e < p.E) {
                    int start, rows;
                    group_rows(p.offsets, e, p.rows_a, &start, &rows);
                    t = (rows + 127) >> 7;
                }
                int incl = t;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
                    if (lane >= d)
                        incl += v;
                }
                if (e <= p.E)
                    tiles_before[e] = carry + incl - t;
                carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
        }
    }
    if constexpr (kFuseX) {
        // the quantizing warps write the token rows of each scale chunk; the
        // other rows of the 128-row chunks stay zero
        // (and of each stage's token codes: only the real rows are written later)
        for (int i = threadIdx.x; i < STAGES * C::SFB_BYTES / 16; i += C::THREADS)
            reinterpret_cast<uint4*>(smem + C::OFF_SFB)[i] = make_uint4(0u, 0u, 0u, 0u);
        for (int i = threadIdx.x; i < STAGES * C::B_BYTES / 16; i += C::THREADS)
            reinterpret_cast<uint4*>(smem + C::OFF_B)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    // Each role sits inside its register branch: with the register split
    // (SPLIT) ptxas then sizes each branch for its own budget.
    if (warp < kFirstEpiWarp) {
        if constexpr (C::SPLIT)
            asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_LOW));
        if (warp == 0) {
            if (lane == 0) {
                // ------------------------------------------------- TMA producer
                uint32_t it = 0;
                bool ok = true;
                // dense: continue from the first item decoded before the wait
                WorkIter wi = kGrouped ? work_begin(p, total_tiles) : first_wi;
                Work w = first_w;
                bool first = !kGrouped && have_first;
                while (ok && (first || work_next(wi, nkb, w))) {
                    const Tile T = first ? first_t : decode_tile<BN, kGrouped>(w.t, p, tiles_before);
                    first = false;
                    if (!T.valid)
                        continue;
                    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                        const int s = static_cast<int>(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (static_cast<int>(it) < npre) {
                            // weight half issued before the dependency wait (first pass over the ring)
                            if constexpr (!kFuseX)
                                stage_loads(s, kb, T, kHalfX, false);
                            continue;
                        }
                        if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kStatusTimeout, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        stage_loads(s, kb, T, kFuseX ? kHalfW : (kHalfW | kHalfX), true);
                    }
                }
            }
        } else if (warp == 1) {
            if (lane == 0) {
                // --------------------------------------------------- MMA issuer
                // W4A8: E4M3 activations, E2M1 weights (the MMA-M side when swapped)
                constexpr uint32_t idesc = kNv   ? idesc_nvf4(BM, BN)
                                           : kA8 ? idesc_mxf8f6f4(BM, BN, kSwap ? kTypeE2M1 : kTypeE4M3,
                                                                  kSwap ? kTypeE4M3 : kTypeE2M1)
                                                 : idesc_mxf4(BM, BN);
                // this one thread's instruction stream paces the tensor pipe: one
                // barrier wait per stage, descriptors from the stage's base
                const uint64_t a_desc = smem_desc(smem_u32(smem + C::OFF_A), 16, 1024, 2);
                const uint64_t b_desc = smem_desc(smem_u32(smem + C::OFF_B), 16, 1024, 2);
                uint32_t it = 0, tcount = 0, pc = 0;
                bool ok = true;
                WorkIter wi = work_begin(p, total_tiles);
                Work w;
                while (ok && work_next(wi, nkb, w)) {
                    const Tile T = decode_tile<BN, kGrouped>(w.t, p, tiles_before);
                    if (!T.valid)
                        continue;
                    // the epilogue must have drained the accumulator of the previous tile
                    // (DualScale: each group's partial buffer is handed over on its own)
                    if (!C::kDual &&
                        !mbar_wait_bounded(accum_empty, (tcount & 1u) ^ 1u, p.status, kStatusTimeout, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                        const int s = static_cast<int>(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        // the scale movers copy a stage's scales only after its full
                        // barrier, so its sf_full barrier implies both
                        if (!mbar_wait_bounded(&sf_full[s], ph, p.status, kStatusTimeout, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const int groups = min(C::GROUPS, p.kb4 - C::GROUPS * kb);
                        uint32_t d_tmem = tmem_base;
                        if constexpr (C::kDual) {
                            // this group's partial buffer must have been read by the epilogue
                            const uint32_t pb = pc & 1u;
                            if (!mbar_wait_bounded(&part_empty[pb], ((pc >> 1) & 1u) ^ 1u, p.status, kStatusTimeout,
                                                   p.wait_ns)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after_sync();
                            d_tmem = tmem_base + pb * BN;
                        }
                        const uint32_t sfa_t = tmem_base + (C::kDual ? 2 : 1) * BN + s * C::SF_COLS;
                        const uint32_t sfb_t = sfa_t + C::SF_COLS_A;
                        const uint64_t ad0 = a_desc + static_cast<uint32_t>((s * C::A_BYTES) >> 4);
                        const uint64_t bd0 = b_desc + static_cast<uint32_t>((s * C::B_BYTES) >> 4);
                        const bool first = C::kDual || kb == w.kb0;
                        // k-th MMA: slab k / 4, 32-byte column k % 4 (64 FP4 or 32 byte
                        // elements); scale chunk k / 2 (MXFP4: bytes 2 (k % 2), +1 of it),
                        // k (NVFP4: all four bytes) or k / 4 (W4A8: byte k % 4)
                        auto mma = [&](int k) {
                            const int slab = k >> 2;
                            const uint64_t ad = ad0 + static_cast<uint32_t>((slab * (BM * kSlabBytes) + 32 * (k & 3)) >> 4);
                            const uint64_t bd = bd0 + static_cast<uint32_t>((slab * (BN * kSlabBytes) + 32 * (k & 3)) >> 4);
                            const uint32_t acc = (first && k == 0) ? 0u : 1u;
                            if constexpr (kNv) {
                                tc_mma_nvf4(tmem_base, ad, bd, idesc, sfa_t + 4 * k, sfb_t + k * C::SF_COLS_B_ATOM, acc);
                            } else if constexpr (kA8) {
                                const int g = k >> 2;
                                tc_mma_mxf8f6f4(tmem_base, ad, bd, idesc_with_sf_id(idesc, static_cast<uint32_t>(k & 3)),
                                                sfa_t + 4 * g, sfb_t + g * C::SF_COLS_B_ATOM, acc);
                            } else {
                                const int g = k >> 1;
                                const uint32_t sf_id = static_cast<uint32_t>(k & 1) * 2u;
                                tc_mma_mxf4(d_tmem, ad, bd, idesc_with_sf_id(idesc, sf_id), sfa_t + 4 * g,
                                            sfb_t + g * C::SF_COLS_B_ATOM, acc);
                            }
                        };
                        if (groups == C::GROUPS) {
#pragma unroll
                            for (int k = 0; k < C::MMAS_PER_GROUP * C::GROUPS; ++k)
                                mma(k);
                        } else {
                            for (int k = 0; k < C::MMAS_PER_GROUP * groups; ++k)
                                mma(k);
                        }
                        tc_commit(&empty[s]);
                        if constexpr (C::kDual) {
                            tc_commit(&part_full[pc & 1u]);
                            ++pc;
                        }
                    }
                    if constexpr (!C::kDual)
                        tc_commit(accum_full);  // also on the abort path: the epilogue never waits on missing MMAs
                    ++tcount;
                }
            }
        } else if (warp < 2 + CPW) {
            if (lane == 0) {
                // ------------------------------------------------ scale movers
                // Copy q of a stage (q = g * (1 + SFB_TILES) + i: i = 0 the
                // MMA-M operand's scale chunk g, i = 1 + j the MMA-N operand's
                // chunk g of row tile j) belongs to warp 2 + q % CPW.
                const int me = warp - 2;
                uint32_t it = 0;
                bool ok = true;
                WorkIter wi = work_begin(p, total_tiles);
                Work w;
                while (ok && work_next(wi, nkb, w)) {
                    const Tile T = decode_tile<BN, kGrouped>(w.t, p, tiles_before);
                    if (!T.valid)
                        continue;
                    for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                        const int s = static_cast<int>(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&full[s], ph, p.status, kStatusTimeout, p.wait_ns)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        const int atoms = min(C::GROUPS, p.kb4 - C::GROUPS * kb) * C::APG;
                        const uint32_t sfa_t = tmem_base + (C::kDual ? 2 : 1) * BN + s * C::SF_COLS;
                        const uint32_t sfb_t = sfa_t + C::SF_COLS_A;
                        const uint32_t sfa_s = smem_u32(smem + C::OFF_SFA + s * C::SFA_BYTES);
                        const uint32_t sfb_s = smem_u32(smem + C::OFF_SFB + s * C::SFB_BYTES);
    #pragma unroll
                        for (int q = me; q < C::ATOMS * (1 + C::SFB_TILES); q += CPW) {
                            const int g = q / (1 + C::SFB_TILES);
                            const int i = q % (1 + C::SFB_TILES);
                            if (g >= atoms)
                                break;
                            if (i == 0)
                                tc_cp_32x128b_warpx4(sfa_t + 4 * g, smem_desc(sfa_s + 512 * g, 0, 128, 0));
                            else
                                tc_cp_32x128b_warpx4(sfb_t + g * C::SF_COLS_B_ATOM + 4 * (i - 1),
                                                     smem_desc(sfb_s + (i - 1) * C::ATOMS * 512 + 512 * g, 0, 128, 0));
                        }
                        tc_commit(&sf_full[s]);  // arrives once this thread's copies have landed
                    }
                }
            }
        }
    } else {
        if constexpr (C::SPLIT)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_HIGH));
        // ------------------------------------------------------ epilogue
        const int ew = warp - kFirstEpiWarp;
        const int quad = warp & 3;  // TMEM lanes 32 * quad ... (a warp reaches only its own quarter)
        const int half = ew >> 2;
        constexpr int CW = C::CW;
        uint8_t* epi = smem + C::OFF_EPI;
        uint32_t tcount = 0;
        uint32_t qit = 0;     // fused: stages this warp has quantized
        bool qok = true;
        bool stored = false;  // this thread has bulk stores in flight
        WorkIter wi = work_begin(p, total_tiles);
        Work w;
        while (work_next(wi, nkb, w)) {
            const Tile T = decode_tile<BN, kGrouped>(w.t, p, tiles_before);
            if (!T.valid)
                continue;
            if constexpr (kFuseX) {
                // ------------------------------------------ token quantization
                // Job j of a stage: lane quarter j % 4 of 32-element block
                // j / 4 (row r, block cl of the stage's K range); 4 consecutive
                // lanes hold one block, as in the activation quantizer.  Only
                // the tile's real token rows are processed: the pad rows of
                // every stage's codes and scale chunks were zeroed at setup
                // and nothing else writes them.  A stage's token loads are all
                // issued before the slot wait (and, for tiles of 16 tokens,
                // one stage ahead), so their latency overlaps.
                constexpr int kBlocksPerRow = C::GROUPS * 4;
                constexpr int kJobs = BN * kBlocksPerRow * 4;
                constexpr int kPer = kJobs / (32 * kEpiWarps);  // jobs per thread per stage
                constexpr int kCh = BN >= 64 ? 2 : (kPer < 4 ? kPer : 4);  // jobs whose loads are in flight together
                static_assert(kJobs % (32 * kEpiWarps) == 0 && kPer % kCh == 0, "whole warps per stage");
                const int et = threadIdx.x - 32 * kFirstEpiWarp;
                const int kbt = p.K / 32;
                const int rows_real = min(BN, p.rows_b - T.n0);
                const int jobs_real = rows_real * kBlocksPerRow * 4;
                // loads of jobs i0 .. i0 + kCh - 1 of stage kb
                auto load_jobs = [&](int kb, int i0, uint4 (&v)[kCh]) {
#pragma unroll
                    for (int i = 0; i < kCh; ++i) {
                        const int j = et + (i0 + i) * 32 * kEpiWarps;
                        const int blk = j >> 2;
                        const int r = blk / kBlocksPerRow;
                        const int cg = kb * kBlocksPerRow + (blk - r * kBlocksPerRow);
                        v[i] = make_uint4(0u, 0u, 0u, 0u);
                        if (j < jobs_real && cg < kbt)
                            v[i] = *reinterpret_cast<const uint4*>(p.x + (static_cast<int64_t>(T.n0) + r) * p.K +
                                                                   static_cast<int64_t>(cg) * 32 + (j & 3) * 8);
                    }
                };
                uint4 vc[kCh], vn[kCh];
                if (w.kb0 < w.kb1)
                    load_jobs(w.kb0, 0, vc);
                for (int kb = w.kb0; kb < w.kb1 && qok; ++kb, ++qit) {
                    const int s = static_cast<int>(qit % STAGES);
                    const uint32_t ph = (qit / STAGES) & 1u;
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kStatusTimeout, p.wait_ns)) {
                        qok = false;
                        break;
                    }
                    uint8_t* bst = smem + C::OFF_B + s * C::B_BYTES;
                    uint8_t* sfb = smem + C::OFF_SFB + s * C::SFB_BYTES;
#pragma unroll 1
                    for (int i0 = 0; i0 < kPer; i0 += kCh) {
                        // the next chunk's loads (or the next stage's first) go out before this one's work
                        if (i0 + kCh < kPer)
                            load_jobs(kb, i0 + kCh, vn);
                        else if (kb + 1 < w.kb1)
                            load_jobs(kb + 1, 0, vn);
#pragma unroll
                        for (int i = 0; i < kCh; ++i) {
                            const int j0 = (et & ~31) + (i0 + i) * 32 * kEpiWarps;  // this warp's first job
                            if (j0 < jobs_real) {  // whole warps together (the lane quantizer shuffles)
                                const int j = j0 + lane;
                                const int q = j & 3;
                                const int blk = j >> 2;
                                const int r = blk / kBlocksPerRow;
                                const int cl = blk - r * kBlocksPerRow;
                                const int cg = kb * kBlocksPerRow + cl;
                                uint4 v = vc[i];
                                if (p.xmul != nullptr && cg < kbt)
                                    v = smooth_bf16x8(v, __ldg(reinterpret_cast<const uint4*>(
                                                             p.xmul + static_cast<int64_t>(cg) * 32 + q * 8)));
                                uint32_t sf;
                                const uint32_t codes = act_quant_lane(v, p.x_uos, sf);
                                if (j < jobs_real && cg < kbt) {
                                    // 128-byte swizzle of the operand stage: 16-byte unit u of row r at u ^ (r % 8)
                                    *reinterpret_cast<uint32_t*>(bst + (cl >> 3) * (BN * kSlabBytes) + r * kSlabBytes +
                                                                 (((cl & 7) ^ (r & 7)) << 4) + q * 4) = codes;
                                    if (q == 0)
                                        sfb[(cl >> 2) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (cl & 3)] =
                                            static_cast<uint8_t>(sf);
                                }
                            }
                        }
#pragma unroll
                        for (int i = 0; i < kCh; ++i)
                            vc[i] = vn[i];
                    }
                    fence_proxy_async_smem();  // the MMA and the scale copies read them through the async proxy
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&full[s]);
                }
            }
            // swapped: this lane's output column has one bias value, an input
            // the MMAs do not touch -- fetch it before the accumulator wait so
            // its latency is not added after the last MMA
            float bias_pre = 0.0f;
            if constexpr (kSwap) {
                const int r = quad * 32 + lane;
                if (p.bias && r < T.rows_valid && w.mode != kPartial)
                    bias_pre = __bfloat162float(p.bias[static_cast<int64_t>(T.expert) * p.ldo + T.a_row0 + r]);
            }
            uint32_t v[CW];
            bool ok = true;
            if constexpr (C::kDual) {
                // DualScale: out = sum over 512-element groups of coarse x the group's
                // partial sum; the partial of group j is read from its TMEM buffer,
                // released, scaled by the group's coarse scale (per weight row: the
                // TMEM lane when swapped, else the output column) and added here
                float accd[CW];
#pragma unroll
                for (int j = 0; j < CW; ++j)
                    accd[j] = 0.0f;
                const int nch = p.K / 512;
                const int r = quad * 32 + lane;
                // swapped: this lane's weight row; normal: lane c holds columns c and c + 32 of the warp's half
                const int64_t crow = kSwap ? T.a_row0 + r : static_cast<int64_t>(T.n0) + half * CW + lane;
                const bool crow_ok = kSwap ? r < T.rows_valid : crow < p.ldo;
                const bool crow2_ok = !kSwap && CW > 32 && crow + 32 < p.ldo;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++tcount) {
                    const float c1 = crow_ok ? __ldg(p.coarse + crow * nch + kb) : 0.0f;
                    const float c2 = crow2_ok ? __ldg(p.coarse + (crow + 32) * nch + kb) : 0.0f;
                    const uint32_t pb = tcount & 1u;
                    ok = ok && mbar_wait_bounded(&part_full[pb], (tcount >> 1) & 1u, p.status, kStatusTimeout, p.wait_ns);
                    tc_fence_after_sync();
                    // the partial in pieces of at most 32 columns (fewer live registers)
                    constexpr int kPc = CW < 32 ? CW : 32;
#pragma unroll
                    for (int c0 = 0; c0 < CW; c0 += kPc) {
                        uint32_t pv[kPc];
                        tmem_load_cols<kPc>(tmem_base + pb * BN + (static_cast<uint32_t>(quad * 32) << 16) + half * CW + c0,
                                            pv);
                        tmem_ld_wait();
#pragma unroll
                        for (int j = 0; j < kPc; ++j) {
                            const float cj = kSwap ? c1 : __shfl_sync(0xFFFFFFFFu, c0 + j < 32 ? c1 : c2, (c0 + j) & 31);
                            accd[c0 + j] = __fmaf_rn(__uint_as_float(pv[j]), cj, accd[c0 + j]);
                        }
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&part_empty[pb]);
                }
#pragma unroll
                for (int j = 0; j < CW; ++j)
                    v[j] = __float_as_uint(accd[j]);
            } else {
                ok = mbar_wait_bounded(accum_full, tcount & 1u, p.status, kStatusTimeout, p.wait_ns);
                tc_fence_after_sync();
                tmem_load_cols<CW>(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * CW, v);
                tmem_ld_wait();
                tc_fence_before_sync();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(accum_empty);  // the accumulator is in registers: let the next tile start
                ++tcount;
            }
            if (!ok)
                break;
            const int r = quad * 32 + lane;
            const __nv_bfloat16* bias = p.bias ? p.bias + static_cast<int64_t>(T.expert) * p.ldo : nullptr;
            uint8_t* stg = epi + ew * C::EPI_WARP_BYTES;  // this warp's staging area
            if (lane == 0 && stored)
                bulk_wait_group_read0();  // the previous store has left the staging area
            __syncwarp();
            if constexpr (kSwap) {
                if (w.mode == kPartial) {
                    // later stages of a split tile: leave the fp32 sums for the
                    // finishing CTA ([BN tokens][128 rows], coalesced per column)
                    float* slot = p.partials + static_cast<int64_t>(blockIdx.x) * (BN * BM);
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        __stcg(slot + (half * CW + j) * BM + r, __uint_as_float(v[j]));
                    __syncwarp();
                    if (lane == 0 && !(p.withhold_signal && blockIdx.x == gridDim.x - 1))
                        red_release_add_gpu(p.flags + blockIdx.x, 1u);  // ready once all 8 warps have added
                    continue;
                }
                if (w.mode == kHead) {
                    // add the partials of the CTAs holding the rest of the tile, in K order
                    const int64_t last_unit = static_cast<int64_t>(w.t + 1) * nkb - 1;
                    const int nparts = unit_owner(last_unit, p.units) - static_cast<int>(blockIdx.x);
                    uint32_t* flags = p.flags + blockIdx.x + 1;
                    // lane j waits for partial j (all in parallel), bounded
                    for (int j = lane; j < nparts; j += 32) {
                        const uint64_t t0 = global_timer_ns();
                        while (ld_acquire_gpu(flags + j) < kEpiWarps) {
                            if (global_timer_ns() - t0 > p.wait_ns) {
                                atomicOr(p.status, kStatusTimeout);
                                break;
                            }
                        }
                    }
                    __syncwarp();
                    // the loads of partial c + 1 are in flight while partial c is added
                    const float* slot = p.partials + static_cast<int64_t>(blockIdx.x + 1) * (BN * BM) + half * CW * BM + r;
                    float nxt[CW];
#pragma unroll
                    for (int j = 0; j < CW; ++j)
                        nxt[j] = nparts > 0 ? __ldcg(slot + j * BM) : 0.0f;
                    for (int c = 0; c < nparts; ++c) {
                        float cur[CW];
#pragma unroll
                        for (int j = 0; j < CW; ++j)
                            cur[j] = nxt[j];
                        if (c + 1 < nparts) {
                            const float* ns = slot + static_cast<int64_t>(c + 1) * (BN * BM);
#pragma unroll
                            for (int j = 0; j < CW; ++j)
                                nxt[j] = __ldcg(ns + j * BM);
                        }
#pragma unroll
                        for (int j = 0; j < CW; ++j)
                            v[j] = __float_as_uint(__uint_as_float(v[j]) + cur[j]);
                    }
                    __syncwarp();
                    // the last of the 8 reading warps puts each counter back to zero
                    for (int j = lane; j < nparts; j += 32)
                        if (atomicAdd(flags + j, 1u) == 2 * kEpiWarps - 1)
                            atomicExch(flags + j, 0u);
                }
                // lane = output column n (weight row); tile columns = tokens.
                // This warp's 32 columns x CW tokens go out as one box,
                // staged as [CW tokens][32 n].
                const float bn = bias_pre;
                __nv_bfloat16* srow = reinterpret_cast<__nv_bfloat16*>(stg) + lane;
#pragma unroll
                for (int j = 0; j < CW; ++j) {
                    float x = __uint_as_float(v[j]);
                    if constexpr (kNv)
                        x *= p.alpha;
                    srow[j * 32] = __float2bfloat16_rn(x + bn);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_2d(&tmO, stg, static_cast<int32_t>(T.a_row0 + quad * 32), T.n0 + half * CW);
                    bulk_commit_group();
                    stored = true;
                }
            } else {
                // lane = output row; this warp's columns n0 + half*CW + [0, CW)
                // go out in 32 x CHUNK chunks through its staging area, in the
                // swizzled layout of the output map (64-byte rows: 16-byte
                // piece q of row i sits at piece position q ^ ((i / 2) % 4);
                // 32-byte rows: q ^ ((i / 4) % 2)), which keeps the rows of
                // one store phase on different banks.
                constexpr int kChunk = C::CHUNK;
                uint8_t* my_row = stg + lane * (kChunk * 2);
                const int rot = kChunk == 32 ? (lane >> 1) & 3 : (lane >> 2) & 1;
                // rows past the end of this expert belong to the next one:
                // there a chunk is stored row by row instead
                const bool whole = !kGrouped || quad * 32 + 31 < T.rows_valid;
#pragma unroll
                for (int c = 0; c < CW; c += kChunk) {
                    const int col0 = T.n0 + half * CW + c;
                    if (whole && c > 0) {
                        if (lane == 0)
                            bulk_wait_group_read0();  // the previous chunk has left the staging area
                        __syncwarp();
                    }
#pragma unroll
                    for (int j = 0; j < kChunk; j += 8) {
                        float f[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            f[i] = __uint_as_float(v[c + j + i]);
                            if constexpr (kNv)
                                f[i] *= p.alpha;
                        }
                        if (bias && col0 + j < p.ldo) {
                            const uint4 bb = *reinterpret_cast<const uint4*>(bias + col0 + j);
                            const uint32_t bw[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                f[2 * i] += __uint_as_float(bw[i] << 16);
                                f[2 * i + 1] += __uint_as_float(bw[i] & 0xFFFF0000u);
                            }
                        }
                        const uint4 o = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                                                   pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
                        if (whole)
                            *reinterpret_cast<uint4*>(my_row + (((j >> 3) ^ rot) << 4)) = o;
                        else if (r < T.rows_valid && col0 + j < p.ldo)
                            *reinterpret_cast<uint4*>(p.out + (T.a_row0 + r) * static_cast<int64_t>(p.ldo) + col0 + j) = o;
                    }
                    if (whole) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmO, stg, col0, static_cast<int32_t>(T.a_row0 + quad * 32));
                            bulk_commit_group();
                            stored = true;
                        }
                    }
                }
            }
        }
        if (stored)
            bulk_wait_group_read0();  // shared memory stays valid until the last store has read it
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

}  // namespace

// --------------------------------------------------------------- host side
// (tensor-map builders and the SM count are shared with the CTA-pair GEMM)
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    });
    return fn;
}

// Operand maps, 128-byte swizzle, one 128-byte shared-memory row per
// operand row and slab:
//   kOpFp4Packed    packed FP4 [rows, K/2] bytes, slab = 128 bytes (256 elements);
//   kOpBytes        E4M3 [rows, K] bytes, slab = 128 bytes (128 elements);
//   kOpFp4Expanded  packed FP4 [rows, K/2] read as 4-bit elements that the TMA
//                   writes 16 to every 16 bytes (low half; 32-byte aligned
//                   base, K % 128 == 0), slab = 128 elements (64 bytes read).
// KC == 1: 2-D boxes of one slab x box_rows.  KC > 1: the rows viewed as
// slabs (3-D), boxes of one slab x box_rows x KC slabs, which land as KC
// consecutive [box_rows][128 B] slabs.
bool make_operand_map(CUtensorMap* map, const void* base, int64_t rows, int64_t K, int box_rows, int kc, int kind)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt =
        kind == kOpFp4Expanded ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const int64_t row_bytes = kind == kOpBytes ? K : K / 2;
    const int64_t slab_elems = kind == kOpFp4Packed ? kSlabBytes : 128;       // box width in map elements
    const int64_t slab_step = kind == kOpFp4Expanded ? 64 : kSlabBytes;       // global bytes per slab
    const int64_t row_elems = kind == kOpFp4Packed ? K / 2 : K;               // map elements per row
    if (kc == 1) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_elems), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(slab_elems), static_cast<cuuint32_t>(box_rows)};
        return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    }
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(slab_elems), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(row_elems / slab_elems)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(slab_step)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(slab_elems), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(kc)};
    return fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// bf16 output [rows, cols] (row stride cols), boxes of box_cols x box_rows
// taken from shared memory with the given swizzle.
bool make_output_map(CUtensorMap* map, void* base, int64_t rows, int64_t cols, int box_cols, int box_rows,
                     CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle, CU_TENSOR_MAP_L2_PROMOTION_NONE,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 148;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 148;
    }
    return cached[dev];
}

namespace {

// Split-K plan of a swapped (M <= 64) problem: S CTAs per tile (S < 2: no
// split) and the workspace that takes.  Split only when at least half the
// SMs would sit idle; S <= 8 keeps the finishing CTA's reduction short, and
// handing the partial sums over through L2 (write, publish, wait, read)
// costs about as much as ten stages, so the split must save more than that.
struct SplitPlan {
    int64_t S;
    size_t bytes;
};

SplitPlan split_plan(int64_t tiles, int64_t nkb, int bn, int sms)
{
    SplitPlan sp{1, 0};
    if (tiles <= 0)
        return sp;
    const int64_t S = std::min<int64_t>(std::min<int64_t>(8, sms / tiles), nkb);
    if (S >= 2 && nkb * (S - 1) >= 10 * S) {
        sp.S = S;
        sp.bytes = (static_cast<size_t>(sms) * 4 + 255) / 256 * 256 + static_cast<size_t>(tiles * S) * bn * BM * 4;
    }
    return sp;
}

// The swapped configuration launch_gemm picks for M <= 64: tile width and
// 256-element slabs per stage.
void swap_config(int64_t M, int64_t K, int* bn, int* kc)
{
    *kc = K % 256 == 0 ? 2 : 1;
    *bn = *kc == 2 ? (M <= 16 ? 16 : M <= 32 ? 32 : 64) : 64;
}

template <int BN, int STAGES, int KC, int CPW, bool kSwap, bool kGrouped, int kFmt = kFmtMx, bool kFuseX = false>
cudaError_t launch_kernel(const GemmArgs& a, cudaStream_t stream)
{
    using C = Cfg<BN, STAGES, KC, CPW, kSwap, kFmt>;
    constexpr bool kNv = C::kNv, kA8 = C::kA8;
    // MMA-M operand / MMA-N operand
    const uint8_t* opA = kSwap ? a.b : a.a;
    const uint8_t* opB = kSwap ? a.a : a.b;
    const int64_t rows_a = kSwap ? a.N : a.M;
    const int64_t rows_b = kSwap ? a.M : a.N;
    CUtensorMap tmA, tmB, tmO;
    // operand kinds: packed FP4 bytes; W4A8: E4M3 bytes (activations) and
    // FP4 expanded by the TMA (weights)
    const int kind_a = kA8 ? (kSwap ? kOpFp4Expanded : kOpBytes) : kOpFp4Packed;
    const int kind_b = kA8 ? (kSwap ? kOpBytes : kOpFp4Expanded) : kOpFp4Packed;
    if (!make_operand_map(&tmA, opA, rows_a, a.K, BM, KC, kind_a))
        return cudaErrorInvalidValue;
    // fused: there is no quantized token operand; the unused B map points at the weights
    if (!make_operand_map(&tmB, kFuseX ? opA : opB, kFuseX ? rows_a : static_cast<int64_t>(a.E) * rows_b, a.K,
                          kFuseX ? BM : BN, KC, kFuseX ? kind_a : kind_b))
        return cudaErrorInvalidValue;
    if (!(kSwap ? make_output_map(&tmO, a.out, a.M, a.N, 32, BN / 2, CU_TENSOR_MAP_SWIZZLE_NONE)
                : make_output_map(&tmO, a.out, a.M, a.N, C::CHUNK, 32,
                                  C::CHUNK == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B)))
        return cudaErrorInvalidValue;
    GemmParams p;
    p.units = 0;
    p.flags = nullptr;
    p.partials = nullptr;
    p.sfa = kSwap ? a.sb : a.sa;
    p.sfb = kSwap ? a.sa : a.sb;
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.offsets = a.row_offsets;
    p.E = a.E;
    p.rows_a = static_cast<int>(rows_a);
    p.rows_b = static_cast<int>(rows_b);
    p.K = static_cast<int>(a.K);
    p.kb4 = static_cast<int>(a.K / 128);
    p.m_tiles = kGrouped ? static_cast<int>((a.M + static_cast<int64_t>(a.E) * 127) / 128)
                         : static_cast<int>((rows_a + 127) / 128);
    p.n_tiles = static_cast<int>((rows_b + BN - 1) / BN);
    p.ldo = static_cast<int>(a.N);
    p.sfb_expert_stride = ((a.N + 127) / 128) * 128 * (a.K / (kNv ? 16 : 32));
    p.alpha = a.alpha;
    p.early_w = (a.early_weights && !kGrouped) ? 1 : 0;
    p.withhold_signal = a.withhold_split_signal ? 1 : 0;
    p.x = static_cast<const uint16_t*>(a.x_bf16);
    p.xmul = static_cast<const uint16_t*>(a.x_mul);
    p.x_uos = a.x_uos;
    p.coarse = a.coarse;
    p.wait_ns = a.wait_ns;
    p.status = a.status;
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (tiles == 0)
        return cudaSuccess;
    const int sms = sm_count();
    int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
    if constexpr (kSwap && !kGrouped) {
        // split-K: S CTAs per tile, each an equal run of the tile's K stages
        const int64_t nkb = (p.kb4 + C::GROUPS - 1) / C::GROUPS;
        const SplitPlan sp = split_plan(tiles, nkb, BN, sms);
        if (sp.S >= 2 && a.workspace && a.workspace_bytes >= sp.bytes) {
            const size_t flag_bytes = (static_cast<size_t>(sms) * 4 + 255) / 256 * 256;
            p.units = tiles * nkb;
            p.flags = static_cast<uint32_t*>(a.workspace);
            p.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(a.workspace) + flag_bytes);
            grid = static_cast<int>(tiles * sp.S);
        }
    }
    const size_t smem = C::SMEM_FIXED + (kGrouped ? sizeof(int32_t) * (a.E + 1) : 0);
    auto kern = gemm_fp4_kernel<BN, STAGES, KC, CPW, kSwap, kGrouped, kFmt, kFuseX>;
    // The shared-memory opt-in is a per-device function attribute: set it
    // once per device (and grow it if a larger grouped prefix needs more).
    // (keyed by context too: a reset device has a new context without it)
    static std::mutex mu;
    static size_t configured[64] = {};
    static unsigned long long configured_ctx[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= 64)
        return err != cudaSuccess ? err : cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long ctx = current_context_id();
        if (configured_ctx[dev] != ctx || configured[dev] < smem) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (err != cudaSuccess)
                return err;
            configured[dev] = smem;
            configured_ctx[dev] = ctx;
        }
        if constexpr (C::SPLIT) {
            // setmaxnreg.inc waits until the registers it asks for are free:
            // never launch a split that the launch's allocation cannot cover
            static int split_ok[64] = {};
            if (split_ok[dev] == 0) {
                cudaFuncAttributes fa;
                err = cudaFuncGetAttributes(&fa, kern);
                if (err != cudaSuccess)
                    return err;
                split_ok[dev] = static_cast<int64_t>(fa.numRegs) * C::THREADS >=
                                        static_cast<int64_t>(C::THREADS / 2) * (C::REGS_LOW + C::REGS_HIGH)
                                    ? 1
                                    : -1;
            }
            if (split_ok[dev] < 0)
                return cudaErrorInvalidConfiguration;
        }
    }
    if (p.units > 0)  // split-K: a tile's first CTA waits for the others
        return launch_coop(kern, dim3(grid), dim3(C::THREADS), smem, stream, tmA, tmB, tmO, p);
    return launch_pdl(kern, dim3(grid), dim3(C::THREADS), smem, stream, tmA, tmB, tmO, p);
}

}  // namespace

size_t gemm_workspace_counter_bytes()
{
    return (static_cast<size_t>(sm_count()) * 4 + 255) / 256 * 256;
}

size_t gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int fmt)
{
    if (M < 1 || M > 64 || N <= 0 || K <= 0 || K % 128 != 0)
        return 0;
    int bn = 0, kc = 0;
    swap_config(M, K, &bn, &kc);
    int groups = 2 * kc;  // 128-element groups of K per stage
    if (fmt == kGemmNv && bn == 16)
        bn = 32;  // launch_gemm_nvfp4 has no 16-token tile
    if (fmt == kGemmW4A8) {
        // launch_gemm_w4a8: two 128-element slabs per stage at any K
        bn = M <= 32 ? 32 : 64;
        groups = 2;
    }
    const int64_t nkb = (K / 128 + groups - 1) / groups;
    return split_plan((N + BM - 1) / BM, nkb, bn, sm_count()).bytes;
}

// NVFP4 operands (dense only): the tile shapes of the MXFP4 path with one
// stage fewer where the doubled scale chunks would overflow shared memory.
cudaError_t launch_gemm_nvfp4(const GemmArgs& a, cudaStream_t stream)
{
    const bool k256 = a.K % 256 == 0;
    if (a.M <= 64) {
        if (!k256)
            return launch_kernel<64, 7, 1, 4, true, false, kFmtNv>(a, stream);
        return a.M <= 32 ? launch_kernel<32, 4, 2, 4, true, false, kFmtNv>(a, stream)
                         : launch_kernel<64, 3, 2, 4, true, false, kFmtNv>(a, stream);
    }
    const bool wide = a.N >= 256 && ((a.M + 127) / 128) * ((a.N + 255) / 256) >= 148;
    if (wide) {
        // twelve scale copies per stage: four scale warps (register split),
        // or two where the split cannot be launched
        const cudaError_t e = launch_kernel<256, 4, 1, 4, false, false, kFmtNv>(a, stream);
        return e == cudaErrorInvalidConfiguration ? launch_kernel<256, 4, 1, 2, false, false, kFmtNv>(a, stream) : e;
    }
    return launch_kernel<128, 5, 1, 4, false, false, kFmtNv>(a, stream);
}

// W4A8: MXFP8 activations x the MXFP4 weights (dense only).  A stage of KC
// slabs covers 128 KC elements of K; the 3-D view needs only K % 128 == 0.
cudaError_t launch_gemm_w4a8(const GemmArgs& a, cudaStream_t stream)
{
    // the expanded FP4 weight tile takes twice its bytes in shared memory:
    // as many stages as fit keep the weight stream in flight
    if (a.M <= 64)
        return a.M <= 32 ? launch_kernel<32, 5, 2, 4, true, false, kFmtA8>(a, stream)
                         : launch_kernel<64, 4, 2, 4, true, false, kFmtA8>(a, stream);
    const bool wide = a.N >= 256 && ((a.M + 127) / 128) * ((a.N + 255) / 256) >= 148;
    if (wide)
        return launch_kernel<256, 4, 1, 2, false, false, kFmtA8>(a, stream);
    return launch_kernel<128, 6, 1, 4, false, false, kFmtA8>(a, stream);
}

// DualScale weights (K % 512 == 0): the MXFP4 tile shapes whose TMEM holds
// two partial buffers beside the scale columns -- 16 / 32 / 64 tokens for
// M <= 64 (weights on the MMA-M side), else 128 x 128 tiles.
cudaError_t launch_gemm_dual(const GemmArgs& a, cudaStream_t stream)
{
    if (a.M <= 64) {
        if (a.M <= 16)
            return launch_kernel<16, 5, 2, 4, true, false, kFmtDual>(a, stream);
        return a.M <= 32 ? launch_kernel<32, 4, 2, 4, true, false, kFmtDual>(a, stream)
                         : launch_kernel<64, 4, 2, 4, true, false, kFmtDual>(a, stream);
    }
    return launch_kernel<128, 3, 2, 4, false, false, kFmtDual>(a, stream);
}

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream)
{
    if (a.fmt == kGemmNv)
        return launch_gemm_nvfp4(a, stream);
    if (a.fmt == kGemmDual)
        return launch_gemm_dual(a, stream);
    if (a.fmt == kGemmW4A8)
        return launch_gemm_w4a8(a, stream);
    // Stages of two slabs need the 3-D operand view, which needs
    // K % 256 == 0; otherwise the one-slab configurations run.
    const bool k256 = a.K % 256 == 0;
    const int64_t m_tiles =
        a.row_offsets != nullptr ? (a.M + static_cast<int64_t>(a.E) * 127) / 128 : (a.M + 127) / 128;
    const bool wide = a.N >= 256 && m_tiles * ((a.N + 255) / 256) >= 148;
    if (a.row_offsets != nullptr) {
        if (wide && a.E <= gemm_pair_max_experts())
            return launch_gemm_pair(a, stream);
        if (wide)
            return launch_kernel<256, 4, 1, 2, false, true>(a, stream);
        return k256 ? launch_kernel<128, 3, 2, 4, false, true>(a, stream)
                    : launch_kernel<128, 6, 1, 4, false, true>(a, stream);
    }
    // decode-sized batches: weights on the 128-row MMA side, tokens as N
    // (the choice swap_config describes)
    if (a.M <= 64 && a.x_bf16 != nullptr) {  // tokens quantized inside the GEMM
        if (!k256)
            return launch_kernel<64, 8, 1, 4, true, false, kFmtMx, true>(a, stream);
        if (a.M <= 16)
            return launch_kernel<16, 5, 2, 4, true, false, kFmtMx, true>(a, stream);
        return a.M <= 32 ? launch_kernel<32, 4, 2, 4, true, false, kFmtMx, true>(a, stream)
                         : launch_kernel<64, 4, 2, 4, true, false, kFmtMx, true>(a, stream);
    }
    if (a.M <= 64) {
        if (!k256)
            return launch_kernel<64, 8, 1, 4, true, false>(a, stream);
        if (a.M <= 16)  // the narrower token slab leaves room for a fifth weight stage
            return launch_kernel<16, 5, 2, 4, true, false>(a, stream);
        return a.M <= 32 ? launch_kernel<32, 4, 2, 4, true, false>(a, stream)
                         : launch_kernel<64, 4, 2, 4, true, false>(a, stream);
    }
    if (wide)
        return a.M >= 256 ? launch_gemm_pair(a, stream) : launch_kernel<256, 4, 1, 2, false, false>(a, stream);
    return k256 ? launch_kernel<128, 3, 2, 4, false, false>(a, stream)
                : launch_kernel<128, 6, 1, 4, false, false>(a, stream);
}

}  // namespace fp4lin
