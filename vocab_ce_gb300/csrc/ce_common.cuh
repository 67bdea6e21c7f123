// ce_common.cuh -- pieces of the vocabulary-parallel cross-entropy shared by
// the translation units that launch it: the shape rules and the kernel that
// combines the per-tile statistics across vocabulary shards.
#pragma once

#include <cuda_runtime.h>

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

// Per token: fold the tiles of each shard into (m_i, s_i), then fold the shards.
__global__ void ce_combine_kernel(const float2 *__restrict__ stats, const float *__restrict__ tau,
                                  const int32_t *__restrict__ targets, int64_t T, int t, int tiles_per_shard,
                                  int v_valid, float *__restrict__ loss, float *__restrict__ lse, uint32_t *err) {
    const int64_t r = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (r >= T) return;
    const int y = targets[r];
    if (y < 0 || y >= v_valid) {
        ptx::record_error(err, kErrInvalid | (1u << 8));
        loss[r] = NAN;
        lse[r] = NAN;
        return;
    }
    float M = -INFINITY, S = 0.0f;
    for (int i = 0; i < t; ++i) {
        // shard i's own statistics, from its vocabulary tiles
        float mi = -INFINITY, si = 0.0f;
        for (int k = 0; k < tiles_per_shard; ++k) {
            const float2 st = stats[static_cast<int64_t>(i * tiles_per_shard + k) * T + r];
            if (st.y > 0.0f) {
                const float nm = fmaxf(mi, st.x);
                si = si * expf(mi - nm) + st.y * expf(st.x - nm);
                mi = nm;
            }
        }
        // the exchange: only (m_i, s_i) crosses shards
        if (si > 0.0f) {
            const float nm = fmaxf(M, mi);
            S = S * expf(M - nm) + si * expf(mi - nm);
            M = nm;
        }
    }
    const float L = M + logf(S);
    lse[r] = L;
    loss[r] = L - tau[r];
}

}  // namespace
}  // namespace tpce
