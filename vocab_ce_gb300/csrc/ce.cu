// ce.cu -- vocab_parallel_ce: the logit GEMM fused with softmax cross-entropy,
// the vocabulary split into t shards laid out on one GPU.
//
// Source: "LIT-022: Megatron-LM ..." (anthology digest), "Key takeaways":
// fuse the parallel logit GEMM into the cross-entropy loss so that each shard
// reduces its logits to per-token numbers and only b*s values are combined,
// not b*s*v logits; the vocabulary is padded so that each shard is a multiple
// of 128 ids.
//
// Forward: one persistent GEMM over all vocabulary tiles of all shards; each
// tile's epilogue reduces its fp32 logits, per token, to (max, sum exp) over
// the real ids and picks up the target logit. A combine kernel folds the
// tiles of a shard into that shard's (m_i, s_i), then folds the shards:
// m = max m_i, S = sum s_i exp(m_i - m), lse = m + ln S, loss = lse - tau.
//
// Backward (the gradient of softmax cross-entropy, dl = g (p - onehot)): the
// vocabulary is walked in chunks that never straddle a shard. For each chunk
// the logits are recomputed and turned into dl (bf16) in a bounded scratch;
// dE_chunk = dl^T H (the shard's own rows) and dH += dl E_chunk (the sum over
// shards, accumulated in fp32 across chunks) follow as two more GEMMs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "ce_common.cuh"
#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

// upper bound of the dl scratch of one vocabulary chunk
constexpr size_t kDlScratchBound = size_t(1) << 30;

struct CeWs {
    int bn;              // vocabulary tile width of the statistics GEMM
    int64_t n_tiles;     // v_pad / bn
    int64_t vc;          // vocabulary chunk width of the backward
    int64_t chunks;      // v_pad / vc
    size_t stats, tau, lse, dl, acc, total;
};

CeWs ce_ws_layout(int64_t T, int64_t h, int64_t v_pad, int t, bool grads) {
    CeWs L{};
    const int64_t vs = v_pad / t;
    L.bn = (vs % 256 == 0) ? 256 : 128;  // a tile never straddles two shards
    L.n_tiles = v_pad / L.bn;
    // chunk = one shard, split into d equal 128-multiples until the scratch fits the bound
    const int64_t q = vs / 128;
    int64_t d = 1;
    while (d < q && (q % d != 0 || static_cast<size_t>(T) * (vs / d) * 2 > kDlScratchBound)) ++d;
    L.vc = vs / d;
    L.chunks = v_pad / L.vc;
    size_t off = 0;
    L.stats = off;
    off = round_up(off + static_cast<size_t>(L.n_tiles) * T * sizeof(float2), 256);
    L.tau = off;
    off = round_up(off + static_cast<size_t>(T) * sizeof(float), 256);
    L.lse = off;
    off = round_up(off + static_cast<size_t>(T) * sizeof(float), 256);
    L.dl = off;
    if (grads) off = round_up(off + static_cast<size_t>(T) * L.vc * 2, 256);
    L.acc = off;
    if (grads && L.chunks > 1) off = round_up(off + static_cast<size_t>(T) * h * sizeof(float), 256);
    L.total = off;
    return L;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_ce_workspace_bytes(int64_t T, int64_t h, int64_t v_pad, int t, int dtype, int with_grads) {
    if (check_ce_shape(T, h, v_pad, 1, t, dtype) != TPCE_OK) return 0;
    return ce_ws_layout(T, h, v_pad, t, with_grads != 0).total;
}

extern "C" tpce_status vocab_parallel_ce(const void *H, const void *E, const int32_t *targets, int64_t T, int64_t h,
                                         int64_t v_pad, int64_t v_valid, int t, float grad_scale, int dtype,
                                         float *loss, float *lse, void *dH, void *dE, void *ws, size_t ws_bytes,
                                         void *stream) {
    tpce_status st = check_ce_shape(T, h, v_pad, v_valid, t, dtype);
    if (st != TPCE_OK) return st;
    if (!E || (T > 0 && (!H || !targets || !loss))) return TPCE_ERR_INVALID;
    for (const void *p : {H, E, static_cast<const void *>(dH), static_cast<const void *>(dE),
                          static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    for (const void *p : {static_cast<const void *>(targets), static_cast<const void *>(loss),
                          static_cast<const void *>(lse)})
        if (reinterpret_cast<uintptr_t>(p) & 3u) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool grads = dH || dE;
    if (T == 0) {
        if (dE && cudaMemsetAsync(dE, 0, static_cast<size_t>(v_pad) * h * 2, s) != cudaSuccess)
            return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const CeWs L = ce_ws_layout(T, h, v_pad, t, grads);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    uint8_t *w = static_cast<uint8_t *>(ws);
    float2 *stats = reinterpret_cast<float2 *>(w + L.stats);
    float *tau = reinterpret_cast<float *>(w + L.tau);
    float *lse_buf = lse ? lse : reinterpret_cast<float *>(w + L.lse);
    __nv_bfloat16 *dl = reinterpret_cast<__nv_bfloat16 *>(w + L.dl);
    float *acc = reinterpret_cast<float *>(w + L.acc);
    uint32_t *err = device_error_word();
    if (!err) return TPCE_ERR_CUDA;
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), vpi = static_cast<int>(v_pad);
    const int vvi = static_cast<int>(v_valid);

    // pass 1: logits of every shard, reduced in the epilogue to per-tile statistics
    {
        Operand a{H, T, h, h};      // K-major [T, h]
        Operand b{E, v_pad, h, h};  // K-major: N = v_pad rows, K = h columns
        EpiCeStats::Params ep{stats, tau, targets, T, vvi, 0, 0};
        st = L.bn == 256
                 ? launch_gemm<256, false, false, EpiCeStats>("ce_fwd_logits_stats", a, b, Ti, vpi, hi, 0, 0, 0, 0, ep, s)
                 : launch_gemm<128, false, false, EpiCeStats>("ce_fwd_logits_stats", a, b, Ti, vpi, hi, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    // exchange of the per-token statistics across shards
    {
        KernelTimer timer("ce_combine", s);
        const int tiles_per_shard = static_cast<int>(L.n_tiles / t);
        ce_combine_kernel<<<static_cast<unsigned>((T + 255) / 256), 256, 0, s>>>(stats, tau, targets, T, t,
                                                                               tiles_per_shard, vvi, loss, lse_buf, err);
        if (check_launch("ce_combine") != TPCE_OK) return TPCE_ERR_CUDA;
    }
    if (!grads) return TPCE_OK;

    const int vci = static_cast<int>(L.vc);
    for (int64_t c = 0; c < L.chunks; ++c) {
        const int n_base = static_cast<int>(c * L.vc);
        // recompute this chunk's logits -> dl = g (softmax - onehot), bf16 scratch
        {
            Operand a{H, T, h, h};
            Operand b{E, v_pad, h, h};  // K-major rows n_base .. n_base + vc
            EpiCeDlogits::Params ep{dl, L.vc, lse_buf, targets, grad_scale, vvi, n_base};
            st = launch_gemm<256, false, false, EpiCeDlogits>("ce_bwd_logits_dl", a, b, Ti, vci, hi, 0, 0, n_base, 0,
                                                               ep, s);
            if (st != TPCE_OK) return st;
        }
        // dE rows of this chunk = dl^T H (no exchange: the rows belong to one shard)
        if (dE) {
            Operand a{dl, T, L.vc, L.vc};  // MN-major: K = T rows, M = vc columns
            Operand b{H, T, h, h};         // MN-major: K = T rows, N = h columns
            EpiStore::Params ep{static_cast<__nv_bfloat16 *>(dE) + static_cast<int64_t>(n_base) * h, nullptr, h};
            st = launch_gemm<256, true, true, EpiStore>("ce_bwd_dE", a, b, vci, hi, Ti, 0, 0, 0, 0, ep, s);
            if (st != TPCE_OK) return st;
        }
        // dH += dl E_chunk: the sum over shards (and chunks), fp32 across launches
        if (dH) {
            Operand a{dl, T, L.vc, L.vc};  // K-major [T, vc]
            Operand b{E, v_pad, h, h};     // MN-major: K = v rows (from n_base), N = h columns
            const int mode = L.chunks == 1 ? 3 : (c == 0 ? 0 : (c == L.chunks - 1 ? 2 : 1));
            EpiAccF32::Params ep{acc, static_cast<__nv_bfloat16 *>(dH), h, mode};
            st = launch_gemm<256, false, true, EpiAccF32>("ce_bwd_dH_shard_sum", a, b, Ti, hi, vci, 0, 0, 0, n_base,
                                                           ep, s);
            if (st != TPCE_OK) return st;
        }
    }
    return TPCE_OK;
}
