// The pair form of the library's GEMM: a cluster of two CTAs on neighbouring
// SMs shares each 256 x 256 output tile through one tcgen05.mma of M = 256
// (cta_group::2), issued by rank 0.  Each CTA loads its own 128 rows of A
// and its own half of B (128 of the tile's 256 columns), so a 64-element K
// slice costs each SM 32 KB of shared memory and L2 traffic instead of the
// single-CTA form's 48 KB, and the ring is 6 stages deep instead of 4.
// grad_X with 256 x 512 tiles (MODE_GRADX_W) issues two such MMAs per K step
// into one 512-column accumulator, from 48 KB slices in a 4-stage ring;
// grad_W shares 7 slots of 32 KB between its ring and its epilogue buffers.
//
//   warp 0 (one lane, both CTAs): TMA producer of the CTA's own halves.
//          Both CTAs' copies of a slice complete on rank 0's `full` barrier
//          (the pair form of the TMA load), which rank 0 arms for both.
//   warp 1 (one lane, rank 0): MMA issuer.  Commits go to both CTAs'
//          barriers (multicast): `empty` frees the slot in both rings,
//          `tmem_full` starts both epilogues.
//   warps 2..9 (both CTAs): the epilogue of the CTA's 128 rows, the same
//          code as the single-CTA form; each warp hands the accumulator back
//          by arriving on rank 0's `tmem_empty`.
//
// Every wait is bounded.  A wait that runs out raises the status bit and
// both CTAs' abort flags; before exiting, each CTA waits (bounded) until the
// MMAs' completion signals for its ring have arrived and the peer has
// finished, so that no signal or read reaches a CTA that has exited.
#pragma once

#include "lce_gemm.cuh"

namespace lce {

struct SharedCtlPair {
    uint64_t full[PAIR_STAGES];
    uint64_t empty[PAIR_STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t fin;
    uint64_t old_full[EPI_WARPS][GRADW_PAIR_BUFS_MAX];  // grad_W (acc_tma 2): an old accumulator block has landed
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(SharedCtlPair) <= CTL_BYTES, "pair control block too large");

// wait_phase of the pair form: running out also raises the peer's abort
// flag.  The acquire stays at CTA scope: these barriers order TMA copies,
// MMAs and TMEM reads, and no wait here orders data the peer's threads wrote.
__device__ __forceinline__ bool wait_phase_pair(uint32_t bar, uint32_t parity, SharedCtlPair* ctl,
                                                uint32_t peer_abort, unsigned* status, uint64_t limit_ns,
                                                bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && ctl->abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            ctl->abort_flag = 1;
            st_shared_cluster_u32(peer_abort, 1u);
            atomicOr(status, STATUS_TIMEOUT);
            return false;
        }
    }
}

// grad_W's read-modify-write of the FP32 accumulator in the chunks between
// the first and the last (acc_tma 2).  Each epilogue warp streams its 32x32
// blocks through its gradw_bufs 4 KB buffers: the old values arrive by
// TMA load that many blocks ahead, the lanes add s times the accumulator in
// place, and a TMA store writes the block back.  Block g of a warp is
// 32-column slab g & 3 of its half of the tile of unit cid + (g >> 2) ncl.
// (Measured on short K loops: the plain loads and stores move the
// accumulator faster than the L2-side adds of acc_tma 1.)
struct OldBlocks {
    float* buf;      // the warp's first buffer
    uint32_t sbuf;   // its shared-memory address
    uint32_t bars;   // the warp's first old_full barrier
    uint32_t nbuf, lg;  // buffers (2 or 4) and log2 of it
    int cid, ncl, num_units, q, half, rank;
    int64_t m_rows;
};

// Coordinates (x = column, y = row) of block g; false past the warp's last tile.
__device__ __forceinline__ bool old_block(const OldBlocks& L, const GemmArgs& a, uint32_t g, int32_t& x,
                                          int32_t& y) {
    const int t = L.cid + static_cast<int>(g >> 2) * L.ncl;
    if (t >= L.num_units) return false;
    int m, n;
    tile_coords(t, a, m, n);
    x = n * BN + 128 * L.half + 32 * static_cast<int>(g & 3);
    y = (2 * m + L.rank) * BM + L.q * 32;
    return true;
}

// Lane 0: the TMA load of block g's old values into its buffer, or for a
// block past the accumulator's rows a plain arrival, so that every block
// completes one phase of its buffer's barrier.
__device__ __forceinline__ void old_issue(const OldBlocks& L, const GemmArgs& a, const CUtensorMap* map, uint32_t g) {
    int32_t x, y;
    if (!old_block(L, a, g, x, y)) return;
    const uint32_t b = g & (L.nbuf - 1);
    const uint32_t bar = L.bars + 8u * b;
    if (y < L.m_rows && LCE_IN((x & 3) == 0 && x < a.N && y >= 0, a.status)) {
        mbar_arrive_expect_tx(bar, EPI_STAGE_FLOATS * 4);
        tma_load_2d(L.sbuf + b * EPI_STAGE_FLOATS * 4, map, bar, x, y);
    } else {
        mbar_arrive(bar);
    }
}

// One tile of the read-modify-write (not inlined: the grad_W epilogue loop
// stays within its registers); g: the warp's next block.  False if a
// wait gave up (the caller drains the loads in flight).
static __device__ __noinline__ bool gradw_tile_old(const GemmArgs& a, const OldBlocks& L, const CUtensorMap* map,
                                               uint32_t& g, uint32_t taddr, int lane, uint32_t empty_bar,
                                               SharedCtlPair* ctl, uint32_t peer_abort, uint64_t limit) {
    const float s = ldexpf(*a.scale, -(P_SCALE_EXP + operand_scale_exp(*a.b_amax_bits)));
    const int j0 = L.half * (BN / 64);
    bool ok = true;
#pragma unroll 1
    for (int jj = 0; jj < BN / 64; ++jj, ++g) {
        int32_t x = 0, y = 0;
        old_block(L, a, g, x, y);
        float v[32];
        tmem_load_32cols(taddr + 32 * (j0 + jj), v);
        const uint32_t b = g & (L.nbuf - 1);
        // (a warp vote keeps the lanes together should their waits end differently)
        if (!__all_sync(0xFFFFFFFFu, wait_phase_pair(L.bars + 8u * b, (g >> L.lg) & 1u, ctl, peer_abort, a.status,
                                                     limit))) {
            ok = false;
            break;
        }
        // the buffer is the TMA box's 128-byte-swizzled layout: row r's
        // 16-byte slot k at slot k ^ (r & 7)
        float* blk = L.buf + b * EPI_STAGE_FLOATS + lane * 32;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            float4* p = reinterpret_cast<float4*>(blk + ((k ^ (lane & 7)) << 2));
            float4 o = *p;
            o.x = fmaf(s, v[4 * k], o.x);
            o.y = fmaf(s, v[4 * k + 1], o.y);
            o.z = fmaf(s, v[4 * k + 2], o.z);
            o.w = fmaf(s, v[4 * k + 3], o.w);
            *p = o;
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            if (y < L.m_rows && LCE_IN((x & 3) == 0 && x < a.N && y >= 0, a.status)) {
                tma_store_2d(map, L.sbuf + b * EPI_STAGE_FLOATS * 4, x, y);
                bulk_commit_group();
            }
            bulk_wait_read_all();  // the store has read the buffer: the next load may fill it
            old_issue(L, a, map, g + L.nbuf);
        }
        __syncwarp();
    }
    tc_fence_before_sync();
    __syncwarp();
    if (lane == 0) release_acc<true>(empty_bar);
    return ok;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(GEMM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c, const GemmArgs args) {
    using T = ModeTraits<MODE>;
    // A chunk without valid rows adds nothing to the grad_W accumulator: unless
    // its tiles overwrite the accumulator (first chunk) or write its bf16 cast
    // (last chunk), every CTA (both of a pair alike) leaves at once.
    if (MODE == MODE_GRADW && gradw_nothing_to_add(args)) return;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1024-byte alignment
    // ring | grad_W block buffers (MODE_GRADW) | control block
    // grad_W: the 7 slots of 32 KB split into 7 - gradw_bufs ring stages and gradw_bufs epilogue buffers per warp
    const int gbufs = (MODE == MODE_GRADW && args.gradw_bufs == 4) ? 4 : 2;
    const int NST = MODE == MODE_GRADW ? GRADW_PAIR_SLOTS - gbufs : (MODE == MODE_GRADX_W ? GRADX_W_STAGES : PAIR_STAGES);
    constexpr int NW = T::NW;                     // 256-column MMAs per output tile
    constexpr int SB = pair_stage_bytes(MODE);    // bytes of one K slice in this CTA
    SharedCtlPair* ctl = reinterpret_cast<SharedCtlPair*>(smem_raw + (base - raw) + pair_ring_bytes(MODE));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = args.timeout_ns;
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    // grad_W epilogue: this warp's block buffer (launched with the extra bytes)
    float* const epi_stage = reinterpret_cast<float*>(smem_raw + (base - raw) + NST * PAIR_STAGE_BYTES) +
                             (warp >= 2 ? (warp - 2) * gbufs * EPI_STAGE_FLOATS : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int w = 0; w < EPI_WARPS; ++w)
            for (int b = 0; b < GRADW_PAIR_BUFS_MAX; ++b) mbar_init(smem_u32(&ctl->old_full[w][b]), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tmem_full[b]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[b]), 2 * EPI_WARPS);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        mbar_init(smem_u32(&ctl->fin), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
        if (MODE == MODE_GRADW && args.acc_tma) tma_prefetch_map(&map_c);
    }
    // Both CTAs' barriers exist before either CTA signals the other.
    __syncwarp();
    cluster_sync_all();
    if (warp == 1) tmem_alloc_pair(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    const uint32_t peer_abort = map_shared_rank(smem_u32(const_cast<int*>(&ctl->abort_flag)), peer);

    const int num_tiles = args.m_tiles * args.n_tiles * (args.k_splits > 1 ? args.k_splits : 1);
    const int cid = static_cast<int>(blockIdx.x >> 1);
    const int ncl = static_cast<int>(gridDim.x >> 1);
    const int dyn = args.dyn_rows ? *args.dyn_rows : -1;
    const int64_t m_rows = (is_gradx(MODE) && dyn >= 0) ? static_cast<int64_t>(dyn) : args.M;
    const int k_blocks = (MODE == MODE_GRADW && dyn >= 0) ? (dyn + BK - 1) / BK : args.k_blocks;
    // grad_X: the last partial round of tiles split over K.  With n fastest in
    // the tile order, the tiles that hold valid rows are the first ones.
    TailPlan tp{num_tiles, 0, 1, k_blocks};
    int num_units = num_tiles;
    if (is_gradx(MODE) && args.tail_out && args.k_splits <= 1 && args.raster == 1) {
        tp = gradx_tail_plan(static_cast<int>((m_rows + PAIR_BM - 1) / PAIR_BM) * args.n_tiles, ncl, k_blocks,
                             TAIL_UNITS_MAX / NW);
        num_units = tp.full + tp.tail * tp.s;
    }

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (this CTA's halves)
            uint32_t stage = 0, phase = 0;
            uint64_t issued = 0;
            bool ok = true;
            for (int t = cid; t < num_units && ok; t += ncl) {
                int m, n, ks, kb0, kb1, tj;
                unit_coords(t, args, tp, k_blocks, m, n, ks, kb0, kb1, tj);
                if (static_cast<int64_t>(m) * PAIR_BM >= m_rows) continue;
                const int32_t arow = m * PAIR_BM + static_cast<int32_t>(rank) * BM;
                // this CTA's half of each 256-column piece of the tile's B
                const int32_t bcol = n * (BN * NW) + static_cast<int32_t>(rank) * (BN / 2);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase_pair(smem_u32(&ctl->empty[stage]), phase ^ 1u, ctl, peer_abort, args.status,
                                         limit)) {
                        ok = false;
                        break;
                    }
                    // rank 0's barrier counts both CTAs' bytes of the slice
                    const uint32_t fb = map_shared_rank(smem_u32(&ctl->full[stage]), 0);
                    if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[stage]), 2 * SB);
                    const uint32_t sa = base + stage * SB;
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    const int32_t k0 = kb * BK;
                    // innermost coordinates: multiples of 8 16-bit elements (16 bytes)
                    (void)LCE_IN((k0 & 7) == 0 && (arow & 7) == 0 && (bcol & 7) == 0, args.status);
                    if constexpr (!T::A_MN) {
                        tma_load_2d_pair(sa, &map_a, fb, k0, args.a_y0 + arow);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d_pair(sa + j * 8192, &map_a, fb, arow + 64 * j, args.a_y0 + k0);
                    }
                    if constexpr (!T::B_MN) {
                        tma_load_2d_pair(sb, &map_b, fb, k0, args.b_y0 + bcol);
                    } else {
#pragma unroll
                        for (int p = 0; p < NW; ++p)
#pragma unroll
                            for (int j = 0; j < (BN / 2) / 64; ++j)
                                tma_load_2d_pair(sb + p * PAIR_B_STAGE_BYTES + j * 8192, &map_b, fb,
                                                 bcol + p * BN + 64 * j, args.b_y0 + k0);
                    }
                    ++issued;
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            const uint64_t last = issued < static_cast<uint64_t>(NST) ? issued : static_cast<uint64_t>(NST);
            if (!ok) {
                // Let this CTA's copies still in flight land before it exits:
                // rank 0 watches them on its barriers (which count both
                // CTAs' bytes); rank 1, whose copies complete there too,
                // gives them a fixed 100 us, far longer than a copy takes.
                if (rank == 0) {
                    for (uint64_t i = 0; i < last; ++i) {
                        const uint64_t j = issued - 1 - i;
                        wait_phase_pair(smem_u32(&ctl->full[j % NST]),
                                        static_cast<uint32_t>((j / NST) & 1u), ctl, peer_abort, args.status,
                                        limit, false);
                    }
                } else {
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 100000ull) {
                    }
                }
            } else {
                // Wait for the MMA completions that free the last slots: they
                // arrive on this CTA's barriers, also from rank 0.
                for (uint64_t i = 0; i < last; ++i) {
                    const uint64_t j = issued - 1 - i;
                    if (!wait_phase_pair(smem_u32(&ctl->empty[j % NST]),
                                         static_cast<uint32_t>((j / NST) & 1u), ctl, peer_abort,
                                         args.status, limit, false))
                        break;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuer (rank 0)
            constexpr uint32_t IDESC = instr_desc_f16kind(PAIR_BM, BN, T::A_MN, T::B_MN, T::F16);
            constexpr uint32_t A_STEP = T::A_MN ? (2048u >> 4) : (32u >> 4);
            constexpr uint32_t B_STEP = T::B_MN ? (2048u >> 4) : (32u >> 4);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = cid; t < num_units && ok; t += ncl) {
                int m, n, ks, kb0, kb1, tj;
                unit_coords(t, args, tp, k_blocks, m, n, ks, kb0, kb1, tj);
                if (static_cast<int64_t>(m) * PAIR_BM >= m_rows) continue;
                if (!wait_phase_pair(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u, ctl, peer_abort, args.status,
                                     limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;  // (acc stays 0 with 512-column tiles)
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase_pair(smem_u32(&ctl->full[stage]), phase, ctl, peer_abort, args.status, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + stage * SB;
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    const uint64_t adesc = T::A_MN ? smem_desc_sw128(sa, 8192, 1024) : smem_desc_sw128(sa, 16, 1024);
#pragma unroll
                    for (int p = 0; p < NW; ++p) {  // piece p: output columns 256 p .. 256 p + 255
                        const uint32_t sbp = sb + p * PAIR_B_STAGE_BYTES;
                        const uint64_t bdesc =
                            T::B_MN ? smem_desc_sw128(sbp, 8192, 1024) : smem_desc_sw128(sbp, 16, 1024);
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_f16kind_pair(d_tmem + p * BN, adesc + A_STEP * k, bdesc + B_STEP * k, IDESC,
                                             (kb != kb0 || k != 0) ? 1u : 0u);
                    }
                    mma_commit_pair_multicast(smem_u32(&ctl->empty[stage]), 0x3);
                    if (++stage == NST) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(smem_u32(&ctl->tmem_full[acc]), 0x3);
                if (NW == 1) acc ^= 1u;  // two accumulators of 256 columns, or one of 512
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                // Wait for every MMA this thread issued before TMEM is freed.
                mma_commit_pair(smem_u32(&ctl->drain));
                wait_phase_pair(smem_u32(&ctl->drain), 0, ctl, peer_abort, args.status, limit, false);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..9) of this CTA's 128 rows
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint32_t acc = 0, acc_phase = 0;
        SideJob side;
        if constexpr (MODE == MODE_LSE)
            side_init(args, side, static_cast<int64_t>(blockIdx.x) * EPI_WARPS + (warp - 2),
                      static_cast<int64_t>(gridDim.x) * EPI_WARPS, (num_tiles - cid + ncl - 1) / ncl);
        // grad_W between the first and the last chunk (acc_tma 2): old blocks by TMA
        const bool old_ldst = MODE == MODE_GRADW && args.acc_tma == 2 && !args.acc_first && !args.write_bf16;
        OldBlocks ob;
        uint32_t og = 0;  // the warp's next block
        if (old_ldst) {
            ob.buf = epi_stage;
            ob.sbuf = smem_u32(epi_stage);
            ob.bars = smem_u32(&ctl->old_full[warp - 2][0]);
            ob.nbuf = static_cast<uint32_t>(gbufs);
            ob.lg = gbufs == 4 ? 2u : 1u;
            ob.cid = cid;
            ob.ncl = ncl;
            ob.num_units = num_units;
            ob.q = q;
            ob.half = half;
            ob.rank = static_cast<int>(rank);
            ob.m_rows = m_rows;
            if (lane == 0)
                for (uint32_t g = 0; g < ob.nbuf; ++g) old_issue(ob, args, &map_c, g);
            __syncwarp();
        }
        bool old_ok = true;
        for (int t = cid; t < num_units; t += ncl) {
            int m, n, ks, kb0, kb1, tj;
            unit_coords(t, args, tp, k_blocks, m, n, ks, kb0, kb1, tj);
            if (static_cast<int64_t>(m) * PAIR_BM >= m_rows) continue;
            const int mc = 2 * m + static_cast<int>(rank);  // this CTA's 128-row tile
            float4 pre[8];
            if constexpr (MODE == MODE_GRADW) {
                const int64_t c0 = static_cast<int64_t>(n) * BN + 128 * half;
                if (gradw_reads_old(args) && c0 < args.N)
                    gradw_load_old(args, static_cast<int64_t>(mc) * BM + q * 32, m_rows, c0, lane, pre);
            }
            // (a warp vote keeps the lanes together should their waits end differently)
            if (!__all_sync(0xFFFFFFFFu, wait_phase_pair(smem_u32(&ctl->tmem_full[acc]), acc_phase, ctl, peer_abort,
                                                         args.status, limit))) {
                old_ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            if (MODE == MODE_GRADW && old_ldst) {
                if (!gradw_tile_old(args, ob, &map_c, og, taddr, lane,
                                    map_shared_rank(smem_u32(&ctl->tmem_empty[acc]), 0), ctl, peer_abort, limit)) {
                    old_ok = false;
                    break;
                }
            } else {
                epilogue_tile<MODE, true>(args, mc, n, q, half, lane, taddr,
                                          map_shared_rank(smem_u32(&ctl->tmem_empty[acc]), 0), m_rows, kb1 <= kb0,
                                          ks, pre, epi_stage, &map_c, tj);
            }
            if (NW == 1) acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
            if constexpr (MODE == MODE_LSE) side_work(args, side, lane, side.budget);
        }
        if constexpr (MODE == MODE_LSE) side_work(args, side, lane, side.units);
        // A wait that gave up (or an abort) leaves loads of old blocks in
        // flight: let them land (bounded waits) before the CTA exits.
        if (MODE == MODE_GRADW && old_ldst && !old_ok) {
            for (uint32_t g = og; g < og + ob.nbuf; ++g) {
                int32_t x, y;
                if (!old_block(ob, args, g, x, y)) break;
                wait_phase_pair(ob.bars + 8u * (g & (ob.nbuf - 1)), (g >> ob.lg) & 1u, ctl, peer_abort,
                                args.status, limit, false);
            }
        }
    }

    __syncwarp();  // reconverge the producer and MMA warps (one lane worked)
    // the epilogue's tile stores/adds read this CTA's shared memory until done
    if (MODE == MODE_GRADW && warp >= 2 && lane == 0) bulk_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    // Neither CTA leaves (or frees TMEM) before the other is done with it.
    if (threadIdx.x == 0) {
        mbar_arrive_cluster(map_shared_rank(smem_u32(&ctl->fin), peer));
        wait_phase_pair(smem_u32(&ctl->fin), 0, ctl, peer_abort, args.status, limit, false);
    }
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

template <int MODE>
cudaError_t launch_gemm_pair(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                             const GemmArgs& args, int grid, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // bit d: shared-memory limit raised on device d
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (grid <= 0 || (grid & 1)) return cudaErrorInvalidConfiguration;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gemm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes(MODE, true));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    gemm_pair_kernel<MODE><<<grid, GEMM_THREADS, gemm_smem_bytes(MODE, true), stream>>>(map_a, map_b, map_c, args);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_gemm_mode(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                             const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    if constexpr (MODE == MODE_GRADX_W) {  // 512-column tiles exist in the pair form only
        return pair ? launch_gemm_pair<MODE>(map_a, map_b, map_c, args, grid, stream) : cudaErrorInvalidValue;
    } else {
        return pair ? launch_gemm_pair<MODE>(map_a, map_b, map_c, args, grid, stream)
                    : launch_gemm_single<MODE>(map_a, map_b, map_c, args, grid, stream);
    }
}

}  // namespace lce
