// gemm_pair.cuh -- the CTA-pair form of the tensor-core GEMM (bf16 operands).
//
// Two CTAs of a cluster share one 256 x BN output tile: the even CTA's MMA
// thread issues tcgen05.mma.cta_group::2, which multiplies each CTA's own 128
// rows of A by the full BN columns of B -- half of B held in each CTA's shared
// memory -- into each CTA's own tensor memory. Per SM a pipeline stage holds
// 128 rows of A and BN/2 rows of B (32 KB at BN = 256 instead of 48 KB), so
// six stages fit and each SM reads a third less from L2 for the same FLOPs;
// the one-CTA kernel is latency-bound on exactly those operand loads.
//
// Signalling between the two CTAs:
//   full[s]    lives in the even CTA; both CTAs' TMA loads count their bytes
//              on it (cp.async.bulk.tensor .cta_group::2 to the even CTA's
//              barrier); the even CTA's producer arms it with both CTAs' bytes.
//   empty[s]   in each CTA, arrived by the even CTA's MMA commit (multicast).
//   tfull[a]   in each CTA, arrived by the even CTA's MMA commit (multicast).
//   tempty[a]  lives in the even CTA; the epilogue warps of both CTAs arrive.
// The epilogue is the one-CTA kernel's, applied to each CTA's 128 rows.
//
// Split tail. When the last wave holds few tiles (host's choice, see
// launch_gemm_pair), each of them is split along K into parts run by
// otherwise idle clusters; a cluster runs at most one part. A part's
// epilogue writes its fp32 partial (per CTA: 128 rows x BN) to global
// scratch, and its four epilogue warps meet on a shared-memory barrier
// (bounded waits) before one thread takes a ticket with an atomic add. The
// part that draws the last ticket sums the partials in part order and runs
// the ordinary epilogue on the sum; no CTA ever waits for another.
#pragma once

#include "gemm.cuh"

namespace tpce {
namespace {

template <int BN, class Epi>
struct PairCfg {
    static_assert(BN == 128 || BN == 256, "pair tile width");
    static constexpr uint32_t kABytes = kBM * kRowBytes;        // this CTA's 128 rows of A
    static constexpr uint32_t kBBytes = (BN / 2) * kRowBytes;   // this CTA's half of B
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kStagingBytes = EpiSmem<Epi>::kBytes;
    static constexpr uint32_t kFree = kSmemMax - 1024 - kBarrierBytes - kStagingBytes;
    static constexpr int kStages = (kFree / kStageBytes) > 6 ? 6 : static_cast<int>(kFree / kStageBytes);
    static_assert(kStages >= 3, "too few pipeline stages");
    static constexpr uint32_t kTmemCols = 2 * BN <= 256 ? 256 : 512;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kStagingBytes + 1024 + kBarrierBytes;
};

template <int BN, bool A_MN, bool B_MN, class Epi, int kChunk>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(64 + 32 * Epi::kWarps, 1)
    tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                        const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ ChunkSet<kChunk> cs,
                        const GemmShape shp, const typename Epi::Params ep, uint32_t *err) {
    using C = PairCfg<BN, Epi>;
    using ET = ElemTraits<__nv_bfloat16>;
    static_assert(Epi::kWarps == 4, "pair epilogue: one warp per TMEM lane quarter");
    constexpr int S = C::kStages;
    constexpr int kBK = ET::kBK;
    constexpr int kUmmaK = ET::kUmmaK;
    constexpr int kHalfN = BN / 2;
    constexpr uint32_t kIdesc = ptx::idesc_f32acc(2 * kBM, BN, ET::kFmt, A_MN, B_MN);
    constexpr int kTileN = Epi::kGated ? BN / 2 : BN;  // output columns per tile
    constexpr int kChunks = kTileN / 32;
    constexpr int kOuts = Epi::kOuts;
    static_assert(!Epi::kGated || BN % 128 == 0, "gated tiles: halves of whole 64-wide blocks");
    static_assert(!(Epi::kGated && kChunk == kChunkB), "gated tiles read an unchunked B");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = smem + S * C::kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(staging + C::kStagingBytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *in_bars = drain + 1;  // 2 per epilogue warp
    uint64_t *tail_bar = in_bars + 2 * Epi::kWarps;  // the epilogue warps' partials are written
    uint64_t *tail_done = tail_bar + 1;             // the ticket is drawn
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tail_done + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile uint32_t *tail_ticket = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();  // 0: the even CTA, which issues the MMAs

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&tfull[i], 1);
            ptx::mbar_init(&tempty[i], 2 * Epi::kWarps);
        }
        for (int i = 0; i < 2 * Epi::kWarps; ++i) ptx::mbar_init(&in_bars[i], 1);
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(tail_bar, Epi::kWarps);
        ptx::mbar_init(tail_done, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if constexpr (kChunk == kChunkA || kChunk == kChunkB) prefetch_chunk_maps(cs);
    }
    if constexpr (kChunk == kChunkC) {
        if (warp == 2 && lane == 0) prefetch_chunk_maps(cs);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // both CTAs' barriers exist before either signals the other
    ptx::cluster_sync();

    const int num_units = shp.full_units + shp.tail_tiles * shp.split;  // tiles of 256 x BN, or their K parts
    const int cluster_id = blockIdx.x >> 1;
    const int clusters = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            uint32_t issued_parity = 0;
            const bool hint = shp.l2_hint != 0;
            const uint64_t pol_a = hint ? ptx::l2_policy_evict_last() : 0;
            const uint64_t pol_b = hint ? ptx::l2_policy_evict_first() : 0;
            auto load = [&](void *dst, const CUtensorMap *m, uint32_t bar, int c0, int c1, uint64_t pol) {
                if (hint)
                    ptx::tma_load_2d_pair_hint(dst, m, bar, c0, c1, pol);
                else
                    ptx::tma_load_2d_pair(dst, m, bar, c0, c1);
            };
            for (int u = cluster_id; u < num_units && !*abort_flag; u += clusters) {
                int tile, kb0, kb1, part;
                unit_coords(u, shp, tile, kb0, kb1, part);
                int mb, rb;
                tile_coords(tile, shp, mb, rb);
                const int m0 = mb * (2 * kBM) + static_cast<int>(rank) * kBM;
                for (int i = 0; i < shp.run_len && !*abort_flag; ++i) {
                    const int nb = rb * shp.run_len + i;
                    // this CTA's half of the B tile; gated tiles: the even CTA loads
                    // the gate columns, the odd CTA the same columns of the up half
                    const int nh0 = Epi::kGated ? nb * kTileN + static_cast<int>(rank) * shp.b_gate_off
                                                : nb * BN + static_cast<int>(rank) * kHalfN;
                    ChunkCursor<kChunk> cur;
                    if constexpr (kChunk == kChunkA) cur.init(cs, A_MN ? shp.a_off_k + kb0 * kBK : m0 + shp.a_off_mn);
                    if constexpr (kChunk == kChunkB) cur.init(cs, B_MN ? shp.b_off_k + kb0 * kBK : nh0 + shp.b_off_mn);
                    // failure-path test knob (off in every ordinary launch): cluster
                    // 0's first tile leaves its first k-block's stage unloaded
                    const int kb_skip = (shp.debug_withhold != 0 && u == 0 && i == 0) ? kb0 : -1;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!ptx::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, 1)) break;
                        const uint32_t bar = ptx::mapa_shared(ptx::smem_u32(&full[stage]), 0);
                        if (rank == 0) ptx::mbar_arrive_expect_tx(&full[stage], 2 * C::kStageBytes);
                        issued |= 1u << stage;
                        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                        uint8_t *sa = smem + stage * C::kStageBytes;
                        uint8_t *sb = sa + C::kABytes;
                        const int k0 = kb * kBK;
                        // outer coordinates: A's M (K-major) or K (MN-major), likewise B's N or K
                        int ya = A_MN ? k0 + shp.a_off_k : m0 + shp.a_off_mn;
                        int yb = B_MN ? k0 + shp.b_off_k : nh0 + shp.b_off_mn;
                        const CUtensorMap *ma = &tmA;
                        const CUtensorMap *mb_ = &tmB;
                        if constexpr (kChunk == kChunkA) {
                            ma = cur.map;
                            ya = cur.y;
                        }
                        if constexpr (kChunk == kChunkB) {
                            mb_ = cur.map;
                            yb = cur.y;
                        }
                        if constexpr ((kChunk == kChunkA && A_MN) || (kChunk == kChunkB && B_MN)) cur.advance(cs, kBK);
                        if (kb != kb_skip) {
                            if (!A_MN) {
                                load(sa, ma, bar, k0 + shp.a_off_k, ya, pol_a);
                            } else {
#pragma unroll
                                for (int j = 0; j < kBM / 64; ++j)
                                    load(sa + j * kMnBlockBytes, ma, bar, m0 + shp.a_off_mn + 64 * j, ya, pol_a);
                            }
                            if (!B_MN) {
                                load(sb, mb_, bar, k0 + shp.b_off_k, yb, pol_b);
                            } else {
#pragma unroll
                                for (int j = 0; j < kHalfN / 64; ++j)
                                    load(sb + j * kMnBlockBytes, mb_, bar, nh0 + shp.b_off_mn + 64 * j, yb, pol_b);
                            }
                        }
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                }
            }
            if (*abort_flag && rank == 0) {
                // the even CTA's full barriers count both CTAs' loads: let them land
                for (int s = 0; s < S; ++s)
                    if (issued & (1u << s)) ptx::mbar_wait_drain(&full[s], (issued_parity >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int u = cluster_id; u < num_units && ok; u += clusters) {
                int tile, kb0, kb1, part;
                unit_coords(u, shp, tile, kb0, kb1, part);
                for (int i = 0; i < shp.run_len; ++i) {
                    if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, err, 2)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * BN;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!ptx::mbar_wait(&full[stage], phase, abort_flag, err, 3)) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        const uint32_t sa = ptx::smem_u32(smem + stage * C::kStageBytes);
                        const uint32_t sb = sa + C::kABytes;
#pragma unroll
                        for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                            const uint64_t ad = A_MN ? ptx::sdesc_sw128(sa + kk * (kUmmaK * kRowBytes), kMnBlockBytes, 1024)
                                                     : ptx::sdesc_sw128(sa + kk * 32, 16, 1024);
                            const uint64_t bd = B_MN ? ptx::sdesc_sw128(sb + kk * (kUmmaK * kRowBytes), kMnBlockBytes, 1024)
                                                     : ptx::sdesc_sw128(sb + kk * 32, 16, 1024);
                            ptx::mma_bf16_pair(d_tmem, ad, bd, kIdesc, ((kb - kb0) | kk) != 0 ? 1u : 0u);
                        }
                        ptx::mma_commit_pair(&empty[stage]);
                        if (++stage == S) {
                            stage = 0;
                            phase ^= 1;
                        }
                    }
                    if (!ok) break;
                    ptx::mma_commit_pair(&tfull[acc]);
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1;
                }
            }
            ptx::mma_commit_pair(drain);
            ptx::mbar_wait_drain(drain, 0);
        }
    } else {
        // ------------------------------------------------ epilogue warps (both CTAs)
        const int ew = warp - 2;
        const int quarter = warp & 3;
        EpiWarp w{staging + ew * EpiSmem<Epi>::kWarpBytes, in_bars + 2 * ew, 0, false, 0u, 0u};
        int acc = 0;
        uint32_t acc_phase = 0;
        bool alive = true;
        for (int u = cluster_id; u < num_units && alive; u += clusters) {
            int tile, kb0, kb1, part;
            unit_coords(u, shp, tile, kb0, kb1, part);
            int mb, rb;
            tile_coords(tile, shp, mb, rb);
            const int row0 = mb * (2 * kBM) + static_cast<int>(rank) * kBM + quarter * 32;
            typename Epi::Row rs;  // this thread's row state, carried along the unit's run of tiles
            for (int i = 0; i < shp.run_len; ++i) {
                const int n0 = (rb * shp.run_len + i) * kTileN;
                if (part < 0) epi_issue_input<Epi>(w, ep, &tmIn, lane, n0, row0);
                const bool ok = ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 4);
                if (!__all_sync(0xffffffffu, ok)) {
                    alive = false;
                    break;
                }
                ptx::tc_fence_after();
                const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
                if (part < 0) {
                    if (!epi_tile<Epi, kChunk>(ep, shp, TmemAcc{taddr}, BN / 2, row0, n0, 0, kChunks, lane, w, rs,
                                               i == 0, i == shp.run_len - 1, &tmC0, &tmC1, &tmIn, &cs, abort_flag,
                                               err)) {
                        alive = false;
                        break;
                    }
                } else {
                    // a K part of a tail tile (runs of one tile only): its partial
                    // to global scratch, all BN accumulator columns of this
                    // thread's row, column-major (a warp's 32 rows of one column
                    // are one 128-byte line)
                    const int tl = tile - shp.full_units;
                    const int64_t slot_floats = static_cast<int64_t>(kBM) * BN;
                    float *mine = shp.partial + (static_cast<int64_t>(tl * shp.split + part) * 2 + rank) * slot_floats +
                                  quarter * 32 + lane;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        float v[32];
                        ptx::tmem_ld32(taddr + c * 32, v);
#pragma unroll
                        for (int e = 0; e < 32; ++e) mine[static_cast<int64_t>(c * 32 + e) * kBM] = v[e];
                    }
                    __threadfence();  // the partial is visible GPU-wide before the ticket below
                    // the accumulator is free again
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&tempty[acc]), 0));
                    acc ^= 1;
                    if (acc == 0) acc_phase ^= 1;
                    // the four epilogue warps' partials are written: draw the ticket
                    if (lane == 0) ptx::mbar_arrive(tail_bar);
                    if (ew == 0 && lane == 0) {
                        uint32_t t = 0xffffffffu;
                        if (ptx::mbar_wait(tail_bar, 0, abort_flag, err, 6)) {
                            t = atomicAdd(&shp.tickets[tl * 2 + rank], 1u);
                            __threadfence();
                        }
                        *tail_ticket = t;
                        ptx::mbar_arrive(tail_done);
                    }
                    bool got = lane == 0 ? ptx::mbar_wait(tail_done, 0, abort_flag, err, 7) : true;
                    if (!__all_sync(0xffffffffu, got)) {
                        alive = false;
                        break;
                    }
                    const uint32_t ticket = __shfl_sync(0xffffffffu, lane == 0 ? *tail_ticket : 0u, 0);
                    if (ticket != static_cast<uint32_t>(shp.split - 1)) continue;  // another part finishes the tile
                    __threadfence();  // every part's partial is visible to this CTA
                    if (ew == 0 && lane == 0) shp.tickets[tl * 2 + rank] = 0;  // leave the ticket clear
                    const PartialAcc sum{shp.partial + (static_cast<int64_t>(tl * shp.split) * 2 + rank) * slot_floats +
                                             quarter * 32 + lane,
                                         2 * slot_floats, shp.split};
                    epi_issue_input<Epi>(w, ep, &tmIn, lane, n0, row0);
                    if (!epi_tile<Epi, kChunk>(ep, shp, sum, BN / 2, row0, n0, 0, kChunks, lane, w, rs, true, true,
                                               &tmC0, &tmC1, &tmIn, &cs, abort_flag, err)) {
                        alive = false;
                        break;
                    }
                    continue;
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(ptx::smem_u32(&tempty[acc]), 0));
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
        }
        if (kOuts > 0 && lane == 0) ptx::bulk_wait_all();
        epi_drain_inputs<Epi>(w);
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still read its shared memory or signal it
    ptx::cluster_sync();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, C::kTmemCols);
    }
}

}  // namespace
}  // namespace tpce
