// ce_common.cuh -- pieces of the vocabulary-parallel cross-entropy shared by
// the translation units that launch it: the shape rules and the kernel that
// combines the per-tile statistics across vocabulary shards.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "tpce.h"

namespace tpce {
namespace {

constexpr int64_t kMaxDim = INT_MAX - 1024;  // kernel coordinates are 32-bit

tpce_status check_ce_shape(int64_t T, int64_t h, int64_t v_pad, int64_t v_valid, int t, int dtype) {
    if (dtype != TPCE_BF16 && dtype != TPCE_F32) return TPCE_ERR_INVALID;
    if (T < 0 || h < 8 || t < 1 || v_pad < 1) return TPCE_ERR_SHAPE;
    if (T > kMaxDim || h > kMaxDim || v_pad > kMaxDim) return TPCE_ERR_SHAPE;
    if (h % 8 != 0) return TPCE_ERR_SHAPE;
    if (v_pad % t != 0 || (v_pad / t) % 128 != 0) return TPCE_ERR_SHAPE;  // 128-multiple shards
    if (v_valid < 1 || v_valid > v_pad) return TPCE_ERR_SHAPE;
    // the fp32 path transposes [T, *] and [v_pad, *] matrices with 32-row blocks in grid.y
    if (dtype == TPCE_F32 && ((T + 31) / 32 > 65535 || (v_pad + 31) / 32 > 65535)) return TPCE_ERR_SHAPE;
    return TPCE_OK;
}

// The per-token statistics of pass 1. The combine receives one (max, sumexp)
// pair per shard and token, [t][T]; the logit GEMM may reach a shard's pair
// through parts_per_shard partial pairs, which its epilogue folds (EpiCeStats).
//
// On the CTA-pair kernel (bf16 operands, shards of whole 256-id tiles) a work
// unit of the logit GEMM is a run of consecutive vocabulary tiles of one
// shard and one 256-token row-block; its epilogue carries the running
// (max, sumexp) of each token from tile to tile in registers and stores it
// once. Ideally a run is a whole shard (parts_per_shard = 1: the exchange is
// then exactly one (max, sumexp) per shard and token), but the units are
// spread over the GPU's 76 CTA pairs, and too few long units leave pairs idle
// in the last round (the 129K-vocabulary config has 64 row-blocks x 8 shards =
// 512 units: 6.74 rounds, 4% idle). So each shard is cut into the fewest equal
// parts (a divisor of its tile count) that keep the pairs at least 98.5% busy:
// 9 parts at that config (runs of 7 tiles, 61 rounds of 4608 units), 5 at the
// 8.3B config, 1 wherever the units fit in one round.
// The one-CTA kernel (fp32, or shards that are not whole 256-id tiles) makes
// one part per tile.
// Scratch: the shards' pairs [t][T]; with several parts per shard also the
// parts' pairs [parts][T] and one ticket per 32-token slab and shard.
constexpr int64_t kCePairClusters = 76;  // CTA pairs of a 152-SM GB300 (fixed, so sizes are known on the host)
#ifndef TPCE_CE_MIN_BUSY
#define TPCE_CE_MIN_BUSY 0.985
#endif
constexpr double kCeMinBusy = TPCE_CE_MIN_BUSY;  // build-time tuning knob

struct CeStatsPlan {
    bool pair;            // pass 1 runs on the CTA-pair kernel
    int bn;               // vocabulary tile width
    int run_len;          // tiles per part
    int parts_per_shard;
    int64_t parts;        // t * parts_per_shard
};

inline CeStatsPlan ce_stats_plan(int64_t T, int64_t v_pad, int t, int dtype, bool pair_kernel) {
    CeStatsPlan P{};
    const int64_t vs = v_pad / t;
    const bool whole256 = dtype == TPCE_BF16 && vs % 256 == 0;
    P.bn = whole256 ? 256 : 128;
    P.pair = whole256 && pair_kernel;
    const int64_t tps = vs / P.bn;  // tiles per shard
    P.run_len = 1;
    P.parts_per_shard = static_cast<int>(tps);
    if (P.pair) {
        const int64_t rows = std::max<int64_t>(1, (T + 255) / 256);
        for (int64_t p = 1; p <= tps; ++p) {
            if (tps % p != 0) continue;
            const int64_t units = rows * t * p;
            const int64_t c = std::min<int64_t>(units, kCePairClusters);
            const int64_t rounds = (units + c - 1) / c;
            if (static_cast<double>(units) >= kCeMinBusy * static_cast<double>(rounds * c)) {
                P.parts_per_shard = static_cast<int>(p);
                break;
            }
        }
        P.run_len = static_cast<int>(tps / P.parts_per_shard);
    }
    P.parts = static_cast<int64_t>(t) * P.parts_per_shard;
    return P;
}

// Bytes of the fold's scratch beside the shards' pairs: the parts' pairs and
// the tickets (none with one part per shard).
inline size_t ce_parts_bytes(const CeStatsPlan &P, int64_t T) {
    return P.parts_per_shard > 1 ? static_cast<size_t>(P.parts) * T * 8 : 0;
}
inline size_t ce_ticket_bytes(const CeStatsPlan &P, int64_t T, int t) {
    return P.parts_per_shard > 1 ? static_cast<size_t>((T + 31) / 32) * t * 4 : 0;
}

// (m, s) <- the log-sum-exp fold of (m, s) and (m2, s2): s e^{m - M} + s2 e^{m2 - M}
// with M = max(m, m2). A part with s2 = 0 holds no real id and is skipped.
__device__ __forceinline__ void lse_fold(float &m, float &s, float m2, float s2) {
    if (s2 > 0.0f) {
        const float nm = fmaxf(m, m2);
        s = s * expf(m - nm) + s2 * expf(m2 - nm);
        m = nm;
    }
}

// Per token: fold the shards' (m_i, s_i). A block takes 32 tokens, one per
// lane, so each shard's statistics arrive as one coalesced 256-byte load per
// warp. Its warps take the shards in turn (warp w: shards w, w + kCombineWarps,
// ...), and warp 0 folds the warps' results. (The kernel also folds several
// pairs per shard, parts_per_shard > 1, which the library no longer passes.)
constexpr int kCombineWarps = 8;
__global__ void __launch_bounds__(32 * kCombineWarps)
    ce_combine_kernel(const float2 *__restrict__ stats, const float *__restrict__ tau,
                      const int32_t *__restrict__ targets, int64_t T, int t, int parts_per_shard, int v_valid,
                      float *__restrict__ loss, float *__restrict__ lse, uint32_t *err) {
    __shared__ float2 part[kCombineWarps][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 32 + lane;
    const bool live = r < T;
    float M = -INFINITY, S = 0.0f;
    if (live) {
        for (int i = warp; i < t; i += kCombineWarps) {
            // shard i's own statistics, from its vocabulary tiles
            const float2 *p = stats + static_cast<int64_t>(i) * parts_per_shard * T + r;
            float mi = -INFINITY, si = 0.0f;
            int k = 0;
            for (; k + 4 <= parts_per_shard; k += 4) {
                float2 st[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) st[j] = __ldg(p + static_cast<int64_t>(k + j) * T);
#pragma unroll
                for (int j = 0; j < 4; ++j) lse_fold(mi, si, st[j].x, st[j].y);
            }
            for (; k < parts_per_shard; ++k) {
                const float2 st = __ldg(p + static_cast<int64_t>(k) * T);
                lse_fold(mi, si, st.x, st.y);
            }
            lse_fold(M, S, mi, si);  // the exchange
        }
    }
    part[warp][lane] = make_float2(M, S);
    __syncthreads();
    if (warp != 0 || !live) return;
    for (int w = 1; w < kCombineWarps; ++w) lse_fold(M, S, part[w][lane].x, part[w][lane].y);
    const int y = targets[r];
    if (y < 0 || y >= v_valid) {
        ptx::record_error(err, kErrInvalid | (1u << 8));
        loss[r] = NAN;
        lse[r] = NAN;
        return;
    }
    const float L = M + logf(S);
    lse[r] = L;
    loss[r] = L - tau[r];
}

inline void launch_ce_combine(const float2 *stats, const float *tau, const int32_t *targets, int64_t T, int t,
                              int parts_per_shard, int v_valid, float *loss, float *lse, uint32_t *err,
                              cudaStream_t s) {
    ce_combine_kernel<<<static_cast<unsigned>((T + 31) / 32), 32 * kCombineWarps, 0, s>>>(
        stats, tau, targets, T, t, parts_per_shard, v_valid, loss, lse, err);
}

}  // namespace
}  // namespace tpce
