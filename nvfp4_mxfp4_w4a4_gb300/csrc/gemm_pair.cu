// gemm_pair.cu -- the W4A4 MXFP4 GEMM of large (prefill-shaped) problems on
// CTA pairs.
//
//   out[m, n] = bf16_rne( sum_k A[m, k] * B[n, k] + bias[n] )
//
// Same operation, operands and rules as gemm.cu ("Efficiently Serving NVFP4
// Models on AMD Instinct MI350X/MI355X ... via Online NVFP4 to Quark MXFP4
// Requantization", "Native FP4 matmul": both operands MXFP4 on native
// block-scaled FP4 matrix instructions; bf16 output with a bf16 row bias per
// "W4A4 MXFP4 Quantization", Configuration).
//
// Why pairs: at the FP4 MMA rate (a 128 x 256 x 64 MMA per 128 cycles per
// SM) a single-CTA 128 x 256 tile needs ~96 bytes of operands per cycle per
// SM, and the TMA copies in flight per SM do not deliver that across the
// ~1 us load round trip.  Here two CTAs on two SMs (a cluster of 2) compute
// a 256 x 256 tile with 256-row MMAs (tcgen05 cta_group::2): each CTA loads
// 128 rows of A and 128 rows of B, so an SM needs ~64 bytes per cycle for
// the same MMA rate.
//
// What limits the operand stream (measured on this GPU with an ingest probe
// of all SMs): a bulk-copy instruction holds its issuing thread ~600 cycles
// whatever its size, so one thread delivers at most one copy per ~600 cycles;
// with copies from several threads an SM takes in up to ~67 bytes per cycle.
// So each operand has its own producer thread, copies are large (two slabs,
// 32 KB), the scale factors do not go through the copy engine at all, and
// the epilogue stores few, large boxes.
//
// Per CTA (16 warps, registers split 88 / 168 with setmaxnreg):
//   warp 0, 6   TMA producers of A and of B: per stage one tensor-map load of
//               the CTA's 128 rows (KC slabs of 256 K-elements); both CTAs'
//               loads count on the LEADER's full barrier;
//   warp 1      TMEM: allocated and freed by both CTAs together; in the
//               leader CTA (even rank) lane 0 issues the pair's MMAs, then a
//               multicast commit frees the stage in both CTAs.  This thread's
//               own instructions pace the tensor pipe (a barrier wait costs
//               it a few hundred cycles even when the phase is complete), so
//               it waits once per stage and forms descriptors from
//               precomputed bases;
//   warps 2-5   scale writers: each loads the stage's scale chunks (its A rows'
//               tile and both 128-row B tiles: each CTA's TMEM needs the
//               scales of all 256 B rows) from global memory into registers
//               ahead of time, waits until the stage's TMEM scale columns are
//               free, writes them into its quarter of the TMEM lanes with
//               tcgen05.st (the layout a 32x128b.warpx4 copy would produce)
//               and arrives on the leader's full barrier of the stage, so
//               that the MMA thread waits once per stage; warp 2 also asks
//               L2 for the next tile's scales (the leader's: the weight
//               scales; grouped: each CTA's activation scales);
//   warp 7      idle (it completes the 8-warp low-register half);
//   warps 8-15  epilogue of the CTA's 128 rows: read the accumulator, release
//               it (arrive on the leader's accum_empty) so the next tile's
//               MMAs start, add bias, round to bf16, TMA-store 32 x 64 boxes
//               (one or two in flight per warp).
// Configurations: two-slab stages (K % 256 == 0) in a ring of three, or of
// two with two store boxes in flight per epilogue warp for grouped problems
// with K <= 1024 (their tiles are paced by the stores); one-slab stages in a
// ring of six otherwise.
// Every wait is bounded; on expiry the kernel records a timeout in the status
// word and winds down.
//
// Grouped (MoE experts, "Efficiently Serving NVFP4 Models ...", "Native FP4
// matmul": the experts on MXFP4): expert e owns rows [off[e], off[e+1]) of A
// and its own weight [N, K/2], scale array and bias row.  A pair tile is two
// consecutive 128-row tiles of one expert (the second may lie past the
// expert's rows when it has an odd tile count: its MMA rows are computed
// from whatever rows follow and never stored), walked expert-major.  Each
// CTA derives the walk from the device offsets after the dependency wait
// (exclusive prefixes of the experts' 128-row tile and pair-tile counts in
// shared memory).  An output box whose 32 rows run past the expert's end is
// stored row by row, so no row of the next expert is written.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "formats.cuh"
#include "internal.h"
#include "ptx.cuh"

#ifndef FP4_PAIR_KC
#define FP4_PAIR_KC 2
#endif

namespace fp4lin {
namespace {

constexpr int kRows = 128;   // rows of A and of B each CTA holds per tile
constexpr int kTileN = 256;  // output columns per tile
constexpr int kSlab = 128;   // packed bytes of K per row per slab (256 elements)
constexpr int kEpiWarps = 8;

struct PairParams {
    const uint8_t* sfa;
    const uint8_t* sfb;
    const __nv_bfloat16* bias;
    __nv_bfloat16* out;         // grouped: rows of partial output boxes are stored directly
    const int32_t* offsets;     // grouped: [E + 1] row offsets (device)
    int E;                      // grouped: experts
    int64_t sfb_expert_stride;  // grouped: scale bytes of one expert's weight
    int M;                      // dense: rows of A
    int N;
    int kb4;        // K / 128
    int m_pairs;    // 256-row tiles of A
    int n_tiles;    // 256-column tiles of the output
    int sfa_tiles;  // 128-row scale tiles of A
    int sfb_tiles;  // 128-row scale tiles of B
    unsigned long long wait_ns;
    unsigned int* status;
};

// EPI_BUFS: store boxes each epilogue warp may have in flight (staging
// buffers of one box each).
template <int KC, int STAGES, int EPI_BUFS = 1>
struct PairCfg {
    static constexpr int GROUPS = 2 * KC;  // 128-element groups of K per stage
    static constexpr int A_BYTES = kRows * kSlab * KC;
    static constexpr int B_BYTES = kRows * kSlab * KC;
    static constexpr int CHUNK = 64;  // output columns per store box (128-byte rows)
    static constexpr int EPI_BOX_BYTES = 32 * CHUNK * 2;
    static constexpr int EPI_WARP_BYTES = EPI_BUFS * EPI_BOX_BYTES;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_BYTES;
    static constexpr int OFF_BAR = OFF_EPI + kEpiWarps * EPI_WARP_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 2;
    static constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_PREFIX = OFF_SLOT + 16;   // grouped: 2 (E + 1) int32
    static constexpr int SMEM = OFF_PREFIX + 1024;     // + 1 KB alignment slack (+ the prefixes when grouped)
    static constexpr int SF_COLS_A = 4 * GROUPS;       // TMEM scale columns per stage
    static constexpr int SF_COLS_B = 8 * GROUPS;
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B;
    static constexpr int TMEM_COLS = 512;
    static constexpr int THREADS = 512;
    static constexpr int FIRST_EPI_WARP = 8;
    static constexpr int REGS_LOW = 88;
    static constexpr int REGS_HIGH = 168;
    static_assert((REGS_LOW + REGS_HIGH) * 256 == 65536, "register split must fill the register file");
    static_assert(kTileN + STAGES * SF_COLS <= TMEM_COLS, "TMEM overflow");
    static_assert(OFF_EPI % 1024 == 0, "staging alignment (swizzled store boxes)");
    static_assert(SMEM <= 232448, "shared memory budget");
    // experts whose prefixes still fit
    static constexpr int MAX_E = (232448 - SMEM) / 8 - 1;
};

// One CTA's share of a pair tile.
struct PairTile {
    int64_t a_row0;  // this CTA's first row of A and of the output
    int rows_valid;  // of its 128 rows, those inside the problem (grouped: inside the expert); <= 0: none
    int sfa_rt;      // its 128-row scale tile of A
    int n0;          // first output column
    int expert;
};

template <bool kGrouped>
__device__ __forceinline__ PairTile pair_tile(int t, int rank, const PairParams& p, const int32_t* tiles_before,
                                              const int32_t* pairs_before)
{
    PairTile T;
    if constexpr (kGrouped) {
        // the expert holding pair tile t: pairs_before[lo] * nt <= t < pairs_before[lo + 1] * nt
        const int nt = p.n_tiles;
        int lo = 0, hi = p.E;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pairs_before[mid] * nt <= t)
                lo = mid;
            else
                hi = mid;
        }
        const int pt = pairs_before[lo + 1] - pairs_before[lo];
        const int local = t - pairs_before[lo] * nt;
        const int gl = 2 * (local % pt) + rank;  // this CTA's 128-row tile of the expert
        int start, rows;
        group_rows(p.offsets, lo, p.M, &start, &rows);
        T.expert = lo;
        T.n0 = (local / pt) * kTileN;
        T.a_row0 = start + static_cast<int64_t>(gl) * kRows;
        T.rows_valid = min(rows - gl * kRows, kRows);
        T.sfa_rt = min(tiles_before[lo] + gl, p.sfa_tiles - 1);  // inside the scale array whatever the offsets
    } else {
        const int mp = t % p.m_pairs;
        T.expert = 0;
        T.n0 = (t / p.m_pairs) * kTileN;
        T.sfa_rt = 2 * mp + rank;
        T.a_row0 = static_cast<int64_t>(T.sfa_rt) * kRows;
        T.rows_valid = min(p.M - T.sfa_rt * kRows, kRows);
    }
    return T;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int KC, int STAGES, bool kGrouped, int EPI_BUFS = 1>
__global__ void __launch_bounds__(512, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmO, const PairParams p)
{
    using C = PairCfg<KC, STAGES, EPI_BUFS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    // leader: A and B of both CTAs landed and the scales are in both CTAs' TMEM
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* empty = full + STAGES;       // stage consumed by the pair's MMAs
    uint64_t* accum_full = empty + STAGES;  // the tile's accumulator is complete
    uint64_t* accum_empty = accum_full + 1;                           // leader: both epilogues hold it
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_SLOT);
    int32_t* tiles_before = reinterpret_cast<int32_t*>(smem + C::OFF_PREFIX);  // grouped: [E + 1]
    int32_t* pairs_before = tiles_before + (kGrouped ? p.E + 1 : 0);          // grouped: [E + 1]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = static_cast<int>(blockIdx.x >> 1);
    const int pairs = static_cast<int>(gridDim.x >> 1);
    const int rk = static_cast<int>(rank);
    const int nkb = (p.kb4 + C::GROUPS - 1) / C::GROUPS;  // stages per tile

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1 + 8);  // the leader's A producer (with the bytes) + 4 scale warps x 2 CTAs
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum_full, 1);
        mbar_init(accum_empty, 2 * kEpiWarps);
        fence_mbar_init();
        tma_prefetch_map(&tmA);
        tma_prefetch_map(&tmB);
        tma_prefetch_map(&tmO);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
        tmem_relinquish_pair();
    }
    // both CTAs' barriers exist and TMEM is allocated before anything crosses the pair
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    grid_dependency_wait();
    launch_dependents();
    if constexpr (kGrouped) {
        if (warp == 2) {
            // exclusive prefixes of the experts' 128-row tile and pair-tile counts
            int carry_t = 0, carry_p = 0;
            for (int base = 0; base <= p.E; base += 32) {
                const int e = base + lane;
                int mt = 0;
                if (e < p.E) {
                    int start, rows;
                    group_rows(p.offsets, e, p.M, &start, &rows);
                    mt = (rows + kRows - 1) / kRows;
                }
                const int pt = (mt + 1) >> 1;
                int it = mt, ip = pt;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int vt = __shfl_up_sync(0xFFFFFFFFu, it, d);
                    const int vp = __shfl_up_sync(0xFFFFFFFFu, ip, d);
                    if (lane >= d) {
                        it += vt;
                        ip += vp;
                    }
                }
                if (e <= p.E) {
                    tiles_before[e] = carry_t + it - mt;
                    pairs_before[e] = carry_p + ip - pt;
                }
                carry_t += __shfl_sync(0xFFFFFFFFu, it, 31);
                carry_p += __shfl_sync(0xFFFFFFFFu, ip, 31);
            }
        }
        __syncthreads();
    }
    // pair tiles of the problem (grouped: read from shared memory where needed, so
    // that no extra value stays live into the register-split roles)
    auto total_tiles = [&]() {
        return kGrouped ? *reinterpret_cast<volatile int32_t*>(pairs_before + p.E) * p.n_tiles
                        : p.m_pairs * p.n_tiles;
    };
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t limit = p.wait_ns;

    if (warp < C::FIRST_EPI_WARP) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_LOW));
        if ((warp == 0 || warp == 6) && lane == 0) {
            // ------------------------------------------------ TMA producers
            // warp 0: this CTA's 128 A rows (the leader's also posts the
            // stage's bytes); warp 6: its 128 B rows
            const bool is_a = warp == 0;
            const CUtensorMap* map = is_a ? &tmA : &tmB;
            uint8_t* base = smem + (is_a ? C::OFF_A : C::OFF_B);
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair; t < total_tiles() && ok; t += pairs) {
                const PairTile T = pair_tile<kGrouped>(t, rk, p, tiles_before, pairs_before);
                const int row0 = is_a ? static_cast<int>(T.a_row0) : T.expert * p.N + T.n0 + kRows * rk;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = static_cast<int>(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kStatusTimeout, limit)) {
                        ok = false;
                        break;
                    }
                    // boxes past the end of K or of the rows are zero-filled and still counted
                    if (leader && is_a)
                        mbar_arrive_expect_tx(&full[s], 2u * (C::A_BYTES + C::B_BYTES));
                    uint8_t* dst = base + s * C::A_BYTES;
                    const uint32_t bar = full_leader + 8u * static_cast<uint32_t>(s);
                    if constexpr (KC == 1)
                        tma_load_2d_pair(dst, map, bar, kb * kSlab, row0);
                    else
                        tma_load_3d_pair(dst, map, bar, 0, row0, kb * KC);
                }
            }
        } else if (warp == 1) {
            if (leader && lane == 0) {
                // --------------------------------------------------- MMA issuer
                constexpr uint32_t idesc = idesc_mxf4(2 * kRows, kTileN);
                const uint64_t a_desc = smem_desc(smem_u32(smem + C::OFF_A), 16, 1024, 2);
                const uint64_t b_desc = smem_desc(smem_u32(smem + C::OFF_B), 16, 1024, 2);
                uint32_t it = 0, tcount = 0;
                bool ok = true;
                for (int t = pair; t < total_tiles() && ok; t += pairs) {
                    // both epilogues must hold the previous tile's accumulator
                    if (!mbar_wait_bounded(accum_empty, (tcount & 1u) ^ 1u, p.status, kStatusTimeout, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    for (int kb = 0; kb < nkb; ++kb, ++it) {
                        const int s = static_cast<int>(it % STAGES);
                        const uint32_t ph = (it / STAGES) & 1u;
                        if (!mbar_wait_bounded(&full[s], ph, p.status, kStatusTimeout, limit)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                        // this one thread's instruction stream paces the tensor pipe:
                        // descriptors are the stage's base plus constant offsets
                        const uint32_t sfa_t = tmem_base + kTileN + s * C::SF_COLS;
                        const uint32_t sfb_t = sfa_t + C::SF_COLS_A;
                        const uint64_t ad0 = a_desc + static_cast<uint32_t>((s * C::A_BYTES) >> 4);
                        const uint64_t bd0 = b_desc + static_cast<uint32_t>((s * C::B_BYTES) >> 4);
                        if (C::GROUPS * (kb + 1) <= p.kb4) {
#pragma unroll
                            for (int k = 0; k < 2 * C::GROUPS; ++k) {
                                // k-th MMA (K = 64): slab k / 4, 32-byte column k % 4;
                                // scale chunk k / 2, bytes 2 (k % 2) and 2 (k % 2) + 1
                                const uint32_t off = ((k >> 2) * (kRows * kSlab) + 32 * (k & 3)) >> 4;
                                tc_mma_mxf4_pair(tmem_base, ad0 + off, bd0 + off,
                                                 idesc_with_sf_id(idesc, static_cast<uint32_t>(k & 1) * 2u),
                                                 sfa_t + 4 * (k >> 1), sfb_t + 8 * (k >> 1), (kb | k) != 0 ? 1u : 0u);
                            }
                        } else {
                            const int groups = p.kb4 - C::GROUPS * kb;  // the last, partial stage of K
                            for (int k = 0; k < 2 * groups; ++k) {
                                const uint32_t off = ((k >> 2) * (kRows * kSlab) + 32 * (k & 3)) >> 4;
                                tc_mma_mxf4_pair(tmem_base, ad0 + off, bd0 + off,
                                                 idesc_with_sf_id(idesc, static_cast<uint32_t>(k & 1) * 2u),
                                                 sfa_t + 4 * (k >> 1), sfb_t + 8 * (k >> 1), (kb | k) != 0 ? 1u : 0u);
                            }
                        }
                        tc_commit_pair_multicast(&empty[s], 0x3);
                    }
                    // also on the abort path: the epilogues never wait on MMAs that were not issued
                    tc_commit_pair_multicast(accum_full, 0x3);
                    ++tcount;
                }
            }
        } else if (warp >= 2 && warp < 6) {
            // ---------------------------------------------------- scale writers
            // warp w writes TMEM lanes 32 (w % 4) ... + 31: lane i of the warp
            // takes row i (16 bytes) of every 512-byte scale chunk, which a
            // 32x128b.warpx4 copy would place in each 32-lane quarter.  The
            // chunks of a stage are loaded before the wait for its columns.
            const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t full_leader = mapa_shared(smem_u32(full), 0);
            uint32_t it = 0;
            bool ok = true;
            for (int t = pair; t < total_tiles() && ok; t += pairs) {
                const PairTile T = pair_tile<kGrouped>(t, rk, p, tiles_before, pairs_before);
                const int n0 = T.n0;
                // rows past the problem (the expert) get zero scales; their outputs are not stored
                const bool has_sfa = T.rows_valid > 0;
                const int nsfb = min(2, p.sfb_tiles - n0 / 128);
                const uint8_t* sfa = p.sfa + static_cast<int64_t>(has_sfa ? T.sfa_rt : 0) * p.kb4 * 512 + lane * 16;
                const uint8_t* sfb0 = p.sfb + T.expert * p.sfb_expert_stride +
                                      static_cast<int64_t>(n0 / 128) * p.kb4 * 512 + lane * 16;
                const uint8_t* sfb1 = sfb0 + (nsfb > 1 ? static_cast<int64_t>(p.kb4) * 512 : 0);
                // the weight scales of this tile (first tile only) and of the next
                // one go to L2 ahead of the stage-by-stage loads, which otherwise find
                // them in memory one stage before use (both CTAs read the same two B
                // scale tiles).  Dense problems with many row pairs per column tile
                // skip it: the pairs then work on a few column tiles at a time, and the
                // next tile's scales are already being read by the pairs ahead.
                if (warp == 2 && lane == 0 && (kGrouped || 4 * p.m_pairs <= pairs)) {
                    const uint32_t tile_bytes = static_cast<uint32_t>(p.kb4) * 512u;
                    if (leader && t == pair)
                        bulk_prefetch_l2(sfb0, tile_bytes * static_cast<uint32_t>(nsfb));
                    if (t + pairs < total_tiles()) {
                        const PairTile U = pair_tile<kGrouped>(t + pairs, rk, p, tiles_before, pairs_before);
                        if (leader) {
                            const int un = min(2, p.sfb_tiles - U.n0 / 128);
                            bulk_prefetch_l2(p.sfb + U.expert * p.sfb_expert_stride +
                                                 static_cast<int64_t>(U.n0 / 128) * p.kb4 * 512,
                                             tile_bytes * static_cast<uint32_t>(un));
                        }
                        // grouped: each CTA's own activation scale tile too (the
                        // weights streaming through L2 have evicted it since the
                        // activation quantizer wrote it)
                        if (kGrouped && U.rows_valid > 0)
                            bulk_prefetch_l2(p.sfa + static_cast<int64_t>(U.sfa_rt) * p.kb4 * 512, tile_bytes);
                    }
                }
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int s = static_cast<int>(it % STAGES);
                    const uint32_t ph = (it / STAGES) & 1u;
                    const int groups = min(C::GROUPS, p.kb4 - C::GROUPS * kb);
                    uint4 va[C::GROUPS], vb0[C::GROUPS], vb1[C::GROUPS];
#pragma unroll
                    for (int g = 0; g < C::GROUPS; ++g) {
                        const int64_t off = static_cast<int64_t>(C::GROUPS * kb + g) * 512;
                        const bool in = g < groups;
                        va[g] = (in && has_sfa) ? __ldg(reinterpret_cast<const uint4*>(sfa + off)) : make_uint4(0u, 0u, 0u, 0u);
                        vb0[g] = in ? __ldg(reinterpret_cast<const uint4*>(sfb0 + off)) : make_uint4(0u, 0u, 0u, 0u);
                        vb1[g] = (in && nsfb > 1) ? __ldg(reinterpret_cast<const uint4*>(sfb1 + off))
                                                  : make_uint4(0u, 0u, 0u, 0u);
                    }
                    // the MMAs that read this stage's scale columns last time are done
                    if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kStatusTimeout, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t cols = tmem_base + lane_base + kTileN + s * C::SF_COLS;
#pragma unroll
                    for (int g = 0; g < C::GROUPS; ++g) {
                        tmem_st_32x32b_x4(cols + 4 * g, va[g].x, va[g].y, va[g].z, va[g].w);
                        tmem_st_32x32b_x4(cols + C::SF_COLS_A + 8 * g, vb0[g].x, vb0[g].y, vb0[g].z, vb0[g].w);
                        tmem_st_32x32b_x4(cols + C::SF_COLS_A + 8 * g + 4, vb1[g].x, vb1[g].y, vb1[g].z, vb1[g].w);
                    }
                    tmem_st_wait();
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive_cluster(full_leader + 8u * static_cast<uint32_t>(s));
                }
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_HIGH));
        // ---------------------------------------------------------- epilogue
        const int ew = warp - C::FIRST_EPI_WARP;
        const int quad = warp & 3;  // TMEM lanes 32 * quad ... (a warp reaches only its own quarter)
        const int half = ew >> 2;
        constexpr int CW = kTileN / 2;  // accumulator columns per warp
        constexpr int kChunk = C::CHUNK;
        const uint32_t accum_empty_leader = mapa_shared(smem_u32(accum_empty), 0);
        uint8_t* stg0 = smem + C::OFF_EPI + ew * C::EPI_WARP_BYTES;
        const int rot = lane & 7;  // 128-byte swizzle of the store box: 16-byte piece q of row i at q ^ (i % 8)
        uint32_t tcount = 0;
        uint32_t boxes = 0;  // store boxes this warp has issued
        for (int t = pair; t < total_tiles(); t += pairs) {
            const PairTile T = pair_tile<kGrouped>(t, rk, p, tiles_before, pairs_before);
            const int n0 = T.n0;
            const int row0 = static_cast<int>(T.a_row0) + quad * 32;
            // rows of this warp's 32 that belong to the expert (dense: rows past M are
            // clipped by the store itself)
            const int rv = kGrouped ? T.rows_valid - quad * 32 : 32;
            const __nv_bfloat16* bias = p.bias ? p.bias + static_cast<int64_t>(T.expert) * p.N : nullptr;
            const bool ok = mbar_wait_bounded(accum_full, tcount & 1u, p.status, kStatusTimeout, limit);
            tc_fence_after_sync();
            uint32_t v[CW];
#pragma unroll
            for (int c = 0; c < CW; c += 32)
                tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + half * CW + c, v + c);
            tmem_ld_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive_cluster(accum_empty_leader);  // the accumulator is in registers
            ++tcount;
            if (!ok)
                break;
            if (rv <= 0)
                continue;
            const bool whole = rv >= 32;
#pragma unroll
            for (int c = 0; c < CW; c += kChunk) {
                const int col0 = n0 + half * CW + c;
                // staging buffers in turn; the store that last used this one
                // (EPI_BUFS boxes ago) must have read it
                uint8_t* stg = stg0 + (boxes % EPI_BUFS) * C::EPI_BOX_BYTES;
                uint8_t* my_row = stg + lane * (kChunk * 2);
                if (whole) {
                    if (lane == 0 && boxes >= EPI_BUFS)
                        bulk_wait_group_read<EPI_BUFS - 1>();
                    __syncwarp();
                }
#pragma unroll
                for (int j = 0; j < kChunk; j += 8) {
                    float f[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        f[i] = __uint_as_float(v[c + j + i]);
                    if (bias && col0 + j < p.N) {
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
                    else if (lane < rv && col0 + j < p.N)
                        *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row0 + lane) * p.N + col0 + j) = o;
                }
                if (whole) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmO, stg, col0, row0);
                        bulk_commit_group();
                    }
                    ++boxes;
                }
            }
        }
        if (boxes > 0)
            bulk_wait_group_read<0>();  // shared memory stays valid until the last store has read it
    }

    // both CTAs are done with the pair's barriers, shared memory and TMEM
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, C::TMEM_COLS);
    }
}

template <int KC, int STAGES, bool kGrouped, int EPI_BUFS = 1>
cudaError_t launch_pair(const GemmArgs& a, cudaStream_t stream)
{
    using C = PairCfg<KC, STAGES, EPI_BUFS>;
    const int E = kGrouped ? a.E : 1;
    if (kGrouped && E > C::MAX_E)
        return cudaErrorInvalidValue;
    CUtensorMap tmA, tmB, tmO;
    if (!make_operand_map(&tmA, a.a, a.M, a.K, kRows, KC, kOpFp4Packed) ||
        !make_operand_map(&tmB, a.b, static_cast<int64_t>(E) * a.N, a.K, kRows, KC, kOpFp4Packed) ||
        !make_output_map(&tmO, a.out, a.M, a.N, C::CHUNK, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    PairParams p;
    p.sfa = a.sa;
    p.sfb = a.sb;
    p.bias = static_cast<const __nv_bfloat16*>(a.bias);
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.offsets = a.row_offsets;
    p.E = E;
    p.sfb_expert_stride = (a.N + 127) / 128 * 128 * (a.K / 32);
    p.M = static_cast<int>(a.M);
    p.N = static_cast<int>(a.N);
    p.kb4 = static_cast<int>(a.K / 128);
    p.m_pairs = static_cast<int>((a.M + 255) / 256);
    p.n_tiles = static_cast<int>((a.N + kTileN - 1) / kTileN);
    // grouped: the scale row tiles fp4_sf_bytes_grouped provides for
    p.sfa_tiles = static_cast<int>(kGrouped ? (a.M + static_cast<int64_t>(E) * 127) / 128 : (a.M + 127) / 128);
    p.sfb_tiles = static_cast<int>((a.N + 127) / 128);
    p.wait_ns = a.wait_ns;
    p.status = a.status;
    // grouped: the pair tiles are counted on the device; at most one partial
    // pair tile per expert beyond the dense count
    const int64_t total = static_cast<int64_t>(p.m_pairs + (kGrouped ? E : 0)) * p.n_tiles;
    if (total == 0)
        return cudaSuccess;
    auto kern = gemm_pair_kernel<KC, STAGES, kGrouped, EPI_BUFS>;
    // grouped: the shared-memory opt-in covers the prefixes of MAX_E experts
    constexpr int kSmemMax = C::SMEM + (kGrouped ? 8 * (C::MAX_E + 1) : 0);
    const int smem = C::SMEM + (kGrouped ? 8 * (E + 1) : 0);
    // per device, once: the shared-memory opt-in, the register split check
    // (setmaxnreg.inc waits until the registers it asks for are free: never
    // launch a split the launch's allocation cannot cover) and the number of
    // pairs that fit on the GPU at once
    // (keyed by context too: a reset device has a new context without the opt-in)
    static std::mutex mu;
    static int resident_pairs[64] = {};
    static unsigned long long configured_ctx[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess || dev < 0 || dev >= 64)
        return err != cudaSuccess ? err : cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        const unsigned long long ctx = current_context_id();
        if (resident_pairs[dev] == 0 || configured_ctx[dev] != ctx) {
            configured_ctx[dev] = ctx;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
            if (err != cudaSuccess)
                return err;
            cudaFuncAttributes fa;
            err = cudaFuncGetAttributes(&fa, kern);
            if (err != cudaSuccess)
                return err;
            if (static_cast<int64_t>(fa.numRegs) * C::THREADS <
                static_cast<int64_t>(C::THREADS / 2) * (C::REGS_LOW + C::REGS_HIGH))
                return cudaErrorInvalidConfiguration;
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(2);
            q.blockDim = dim3(C::THREADS);
            q.dynamicSmemBytes = kSmemMax;
            cudaLaunchAttribute qa[1];
            qa[0].id = cudaLaunchAttributeClusterDimension;
            qa[0].val.clusterDim.x = 2;
            qa[0].val.clusterDim.y = 1;
            qa[0].val.clusterDim.z = 1;
            q.attrs = qa;
            q.numAttrs = 1;
            int clusters = 0;
            err = cudaOccupancyMaxActiveClusters(&clusters, kern, &q);
            if (err != cudaSuccess || clusters <= 0)
                return err != cudaSuccess ? err : cudaErrorInvalidConfiguration;
            resident_pairs[dev] = std::min(clusters, sm_count() / 2);
        }
    }
    const int pairs = static_cast<int>(std::min<int64_t>(total, resident_pairs[dev]));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmO, p);
}

}  // namespace

cudaError_t launch_gemm_pair(const GemmArgs& a, cudaStream_t stream)
{
    // stages of two slabs need the 3-D operand view (K % 256 == 0)
    const bool kc2 = FP4_PAIR_KC == 2 && a.K % 256 == 0;
    if (a.row_offsets != nullptr) {
        // short K (at most two stages a tile, as in an MoE down projection): the
        // epilogue's stores, not the operand ring, pace the tiles, so two of the
        // three stages' shared memory go to a second store box per epilogue warp
        if (kc2 && a.K <= 1024)
            return launch_pair<2, 2, true, 2>(a, stream);
        return kc2 ? launch_pair<2, 3, true>(a, stream) : launch_pair<1, 6, true>(a, stream);
    }
    return kc2 ? launch_pair<2, 3, false>(a, stream) : launch_pair<1, 6, false>(a, stream);
}

int gemm_pair_max_experts()
{
    return std::min(std::min(PairCfg<2, 3>::MAX_E, PairCfg<1, 6>::MAX_E), PairCfg<2, 2, 2>::MAX_E);
}

}  // namespace fp4lin
