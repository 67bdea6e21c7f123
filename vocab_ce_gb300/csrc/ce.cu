// ce.cu -- vocab_parallel_ce: the logit GEMM fused with softmax cross-entropy,
// the vocabulary split into t shards laid out on one GPU.
//
// Source: "LIT-022: Megatron-LM ..." (anthology digest), "Key takeaways":
// fuse the parallel logit GEMM into the cross-entropy loss so that each shard
// reduces its logits to per-token numbers and only b*s values are combined,
// not b*s*v logits; the vocabulary is padded so that each shard is a multiple
// of 128 ids.
//
// Forward: one persistent GEMM over all vocabulary tiles of all shards; its
// epilogue reduces the fp32 logits of a run of tiles of one shard, per token,
// to (max, sum exp) over the real ids, carried from tile to tile, and picks up
// the target logit; a shard covered by several runs has their pairs folded by
// the epilogue that finishes last (see ce_stats_plan, EpiCeStats). A combine
// kernel then folds the shards' (m_i, s_i): m = max m_i,
// S = sum s_i exp(m_i - m), lse = m + ln S, loss = lse - tau.
//
// Backward (the gradient of softmax cross-entropy, dl = g (p - onehot)): the
// vocabulary is walked in chunks of whole shards (or parts of one shard). For each chunk
// the logits are recomputed and turned into dl in a bounded scratch;
// dE_chunk = dl^T H (the shard's own rows) and dH += dl E_chunk (the sum over
// shards, accumulated in fp32 across chunks) follow as two more GEMMs.
//
// bf16 tensors read H as the dE GEMM's N operand and E as the dH GEMM's N
// operand in place, and dl^T either in place (MN-major) or, from the hidden
// width below on, from a [vc, T] copy that the dl GEMM's epilogue writes beside
// dl; the fp32 (tf32) path transposes them into the workspace first.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>
#include <cmath>

#include "ce_common.cuh"
#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

// upper bound of the dl scratch of one vocabulary chunk (dl, and its
// transposed copy where dE reads one), build-time tuning knob
#ifndef TPCE_DL_SCRATCH_BOUND
#define TPCE_DL_SCRATCH_BOUND (1ll << 30)
#endif
constexpr size_t kDlScratchBound = static_cast<size_t>(TPCE_DL_SCRATCH_BOUND);

// dE = dl^T H contracts over tokens, and with dl stored [T, vc] its A operand
// is MN-major, which costs the tensor core about 11% against a K-major A
// (measured on GB300). From this hidden width on, the dl GEMM's epilogue also
// stores each dl tile transposed into a [vc, T] copy (a second TMA store of
// the same values, 2 T vc bytes) so that dE reads A K-major. At the 129K
// config that made the dl GEMM about 0.5% slower and took dE from 22.7 to
// about 21 ms per step; a separate transpose pass (4 T vc bytes at HBM speed,
// 1.4 ms per step there) did the same job before.
#ifndef TPCE_DE_KMAJOR_MIN_H
#define TPCE_DE_KMAJOR_MIN_H 6144
#endif
inline bool de_kmajor(int64_t h, int dtype) { return dtype == TPCE_BF16 && h >= TPCE_DE_KMAJOR_MIN_H; }
inline int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }  // bf16 rows padded to 16 bytes

inline int64_t pad4(int64_t x) { return (x + 3) / 4 * 4; }  // fp32 rows padded to 16 bytes

struct CeWs {
    CeStatsPlan plan;    // pass 1's tiles, runs and statistics parts
    int64_t vc;          // vocabulary chunk width of the backward
    int64_t chunks;      // v_pad / vc
    size_t tail, stats, parts, tickets, tau, lse, dl, dlT, acc, Ht, Et, dlt, total;
};

CeWs ce_ws_layout(int64_t T, int64_t h, int64_t v_pad, int t, bool grads, int dtype) {
    CeWs L{};
    const bool f32 = dtype == TPCE_F32;
    const size_t esz = f32 ? 4 : 2;
    const int64_t vs = v_pad / t;
    L.plan = ce_stats_plan(T, v_pad, t, dtype, TPCE_PAIR_BN == 256);  // a tile never straddles two shards
    // chunk = g whole shards: the largest g dividing t with g <= t / 2 (so the
    // whole vocabulary's dl is never resident) whose scratch fits the bound.
    // Fewer, wider chunks mean fewer fp32 passes over the dH accumulator
    // (measured: 1457 -> 1517 TFLOP/s for the 8.3B block going from 1 to 4
    // shards per chunk). When one shard alone is too large, it is split into d
    // equal 128-multiples until the scratch fits.
    // With the transposed copy for dE the scratch holds dl twice.
    const size_t copies = (grads && de_kmajor(h, dtype)) ? 2 : 1;
    const size_t row_bytes = copies * static_cast<size_t>(pad8(T)) * esz;  // per vocabulary id of a chunk
    int64_t g = 1;
    for (int64_t c = 2; c <= t / 2; ++c)
        if (t % c == 0 && row_bytes * (c * vs) <= kDlScratchBound) g = c;
    const int64_t q = vs / 128;
    int64_t d = 1;
    while (d < q && (q % d != 0 || row_bytes * (vs / d) > kDlScratchBound)) ++d;
    L.vc = g > 1 ? g * vs : vs / d;
    L.chunks = v_pad / L.vc;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    L.tail = take(kTailScratchBytes);  // the GEMMs' split tails
    L.stats = take(static_cast<size_t>(t) * T * sizeof(float2));
    L.parts = take(ce_parts_bytes(L.plan, T));
    L.tickets = take(ce_ticket_bytes(L.plan, T, t));
    L.tau = take(static_cast<size_t>(T) * sizeof(float));
    L.lse = take(static_cast<size_t>(T) * sizeof(float));
    if (grads) {
        L.dl = take(static_cast<size_t>(T) * L.vc * esz);
        // the chunk's dl^T [vc, T] (rows padded to 8 tokens) for a K-major dE
        if (de_kmajor(h, dtype)) L.dlT = take(static_cast<size_t>(L.vc) * pad8(T) * esz);
        // bf16: dH accumulates in fp32 over the chunks, then is converted once
        if (!f32) L.acc = take(static_cast<size_t>(T) * h * sizeof(float));
        if (f32) {
            const size_t Tp = static_cast<size_t>(pad4(T));
            L.Ht = take(static_cast<size_t>(h) * Tp * 4);
            L.Et = take(static_cast<size_t>(h) * v_pad * 4);
            L.dlt = take(static_cast<size_t>(L.vc) * Tp * 4);
        }
    }
    L.total = off;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

struct CeArgs {
    const void *H, *E;
    const int32_t *targets;
    int64_t T, h, v_pad, v_valid;
    int t;
    float grad_scale;
    float *loss, *lse;
    void *dH, *dE;
};

// pass 1 + combine, both dtypes
template <typename ElemT>
tpce_status ce_forward(const CeArgs &a, const CeWs &L, void *ws, float *lse_buf, cudaStream_t s) {
    float2 *stats = at<float2>(ws, L.stats);
    float *tau = at<float>(ws, L.tau);
    uint32_t *err = device_error_word();
    if (!err) return fail(TPCE_ERR_CUDA, "vocab_parallel_ce: device status word");
    const int Ti = static_cast<int>(a.T), hi = static_cast<int>(a.h), vpi = static_cast<int>(a.v_pad);
    const int vvi = static_cast<int>(a.v_valid);
    Operand A{a.H, a.T, a.h, a.h};          // K-major [T, h]
    Operand B{a.E, a.v_pad, a.h, a.h};      // K-major: N = v_pad rows, K = h columns
    const CeStatsPlan &P = L.plan;
    uint32_t *tickets = at<uint32_t>(ws, L.tickets);
    const size_t tb = ce_ticket_bytes(P, a.T, a.t);
    if (tb && cudaMemsetAsync(tickets, 0, tb, s) != cudaSuccess)
        return fail(TPCE_ERR_CUDA, "vocab_parallel_ce: cudaMemsetAsync of the statistics tickets");
    EpiCeStats::Params ep{stats, at<float2>(ws, L.parts), tickets, tau, a.targets, a.T, vvi, 0, 0, P.bn, P.run_len,
                          P.parts_per_shard, a.t};
    const TailScratch tail{at<uint8_t>(ws, L.tail), kTailScratchBytes};
    tpce_status st;
    if constexpr (std::is_same<ElemT, __nv_bfloat16>::value && TPCE_PAIR_BN == 256) {
        if (P.pair)
            st = launch_gemm_pair<256, false, false, EpiCeStats>("ce_fwd_logits_stats", A, B, nullptr, nullptr, Ti, vpi, hi,
                                                                 0, 0, 0, 0, ep, s, true, 0, nullptr, &tail, P.run_len);
        else
            st = launch_gemm<ElemT, 128, false, false, EpiCeStats>("ce_fwd_logits_stats", A, B, nullptr, nullptr, Ti, vpi,
                                                                   hi, 0, 0, 0, 0, ep, s);
    } else if (P.bn == 256)
        st = launch_gemm<ElemT, 256, false, false, EpiCeStats>("ce_fwd_logits_stats", A, B, nullptr, nullptr, Ti, vpi, hi, 0,
                                                               0, 0, 0, ep, s);
    else
        st = launch_gemm<ElemT, 128, false, false, EpiCeStats>("ce_fwd_logits_stats", A, B, nullptr, nullptr, Ti, vpi, hi, 0,
                                                               0, 0, 0, ep, s);
    if (st != TPCE_OK) return st;
    // exchange of the per-token statistics across shards
    KernelTimer timer("ce_combine", s);
    launch_ce_combine(stats, tau, a.targets, a.T, a.t, 1, vvi, a.loss, lse_buf, err, s);
    return check_launch("ce_combine", s);
}

tpce_status ce_backward_bf16(const CeArgs &a, const CeWs &L, void *ws, const float *lse_buf, cudaStream_t s) {
    using bf = __nv_bfloat16;
    bf *dl = at<bf>(ws, L.dl);
    float *acc = at<float>(ws, L.acc);
    const TailScratch tail{at<uint8_t>(ws, L.tail), kTailScratchBytes};
    const int Ti = static_cast<int>(a.T), hi = static_cast<int>(a.h), vci = static_cast<int>(L.vc);
    const int vvi = static_cast<int>(a.v_valid);
    for (int64_t c = 0; c < L.chunks; ++c) {
        const int n_base = static_cast<int>(c * L.vc);
        tpce_status st;
        // recompute this chunk's logits -> dl = g (softmax - onehot)
        // at widths where dE reads dl^T, the dl epilogue writes it beside dl
        const bool with_t = a.dE && de_kmajor(a.h, TPCE_BF16);
        {
            Operand A{a.H, a.T, a.h, a.h};
            Operand B{a.E, a.v_pad, a.h, a.h};  // K-major rows n_base .. n_base + vc
            typename EpiCeDlogits<bf>::Params ep{lse_buf, a.targets, a.grad_scale, vvi, n_base};
            if (with_t) {
                const OutView o[2] = {{dl, a.T, L.vc, L.vc}, {at<bf>(ws, L.dlT), L.vc, a.T, pad8(a.T)}};
                st = launch_gemm_auto<bf, false, false, EpiCeDlogitsT, kBN192 | kBN256>(
                    "ce_bwd_logits_dl", A, B, o, nullptr, Ti, vci, hi, 0, 0, n_base, 0, ep, s, 0, nullptr, &tail);
            } else {
                const OutView o[1] = {{dl, a.T, L.vc, L.vc}};
                st = launch_gemm_auto<bf, false, false, EpiCeDlogits<bf>, kBN192 | kBN256>(
                    "ce_bwd_logits_dl", A, B, o, nullptr, Ti, vci, hi, 0, 0, n_base, 0, ep, s, 0, nullptr, &tail);
            }
            if (st != TPCE_OK) return st;
        }
        // dE rows of this chunk = dl^T H (no exchange: the rows belong to one shard)
        if (with_t) {
            bf *dlT = at<bf>(ws, L.dlT);
            const int64_t Tp = pad8(a.T);
            Operand A{dlT, L.vc, a.T, Tp};  // K-major: M = vc rows, K = T columns
            Operand B{a.H, a.T, a.h, a.h};  // MN-major: K = T rows, N = h columns
            const OutView o[1] = {{static_cast<bf *>(a.dE) + static_cast<int64_t>(n_base) * a.h, L.vc, a.h, a.h}};
            st = launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>("ce_bwd_dE", A, B, o, nullptr, vci, hi,
                                                                                   Ti, 0, 0, 0, 0, {nullptr}, s, 0, nullptr,
                                                                                   &tail);
            if (st != TPCE_OK) return st;
        } else if (a.dE) {
            Operand A{dl, a.T, L.vc, L.vc};  // MN-major: K = T rows, M = vc columns
            Operand B{a.H, a.T, a.h, a.h};   // MN-major: K = T rows, N = h columns
            const OutView o[1] = {{static_cast<bf *>(a.dE) + static_cast<int64_t>(n_base) * a.h, L.vc, a.h, a.h}};
            st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>("ce_bwd_dE", A, B, o, nullptr, vci, hi, Ti,
                                                                                  0, 0, 0, 0, {nullptr}, s, 0, nullptr,
                                                                                  &tail);
            if (st != TPCE_OK) return st;
        }
        // dH += dl E_chunk: the sum over shards (and chunks), in fp32, stored by
        // the first chunk and added by the TMA reduction for the others
        if (a.dH) {
            Operand A{dl, a.T, L.vc, L.vc};     // K-major [T, vc]
            Operand B{a.E, a.v_pad, a.h, a.h};  // MN-major: K = v rows (from n_base), N = h columns
            const OutView o[1] = {{acc, a.T, a.h, a.h}};
            st = launch_gemm_auto<bf, false, true, EpiF32Accumulate, kBN192 | kBN256>(
                "ce_bwd_dH_shard_sum", A, B, o, nullptr, Ti, hi, vci, 0, 0, 0, n_base, {c == 0 ? 0 : 1}, s, 0,
                nullptr, &tail);
            if (st != TPCE_OK) return st;
        }
    }
    if (a.dH) return f32_to_bf16(acc, a.dH, a.T * a.h, s);
    return TPCE_OK;
}

tpce_status ce_backward_f32(const CeArgs &a, const CeWs &L, void *ws, const float *lse_buf, cudaStream_t s) {
    float *dl = at<float>(ws, L.dl);
    float *Ht = at<float>(ws, L.Ht), *Et = at<float>(ws, L.Et), *dlt = at<float>(ws, L.dlt);
    const int64_t Tp = pad4(a.T);
    const int Ti = static_cast<int>(a.T), hi = static_cast<int>(a.h), vci = static_cast<int>(L.vc);
    const int vvi = static_cast<int>(a.v_valid);
    tpce_status st;
    if (a.dE && (st = transpose_f32(static_cast<const float *>(a.H), a.T, a.h, a.h, Ht, Tp, s)) != TPCE_OK) return st;
    if (a.dH &&
        (st = transpose_f32(static_cast<const float *>(a.E), a.v_pad, a.h, a.h, Et, a.v_pad, s)) != TPCE_OK)
        return st;
    for (int64_t c = 0; c < L.chunks; ++c) {
        const int n_base = static_cast<int>(c * L.vc);
        {
            Operand A{a.H, a.T, a.h, a.h};
            Operand B{a.E, a.v_pad, a.h, a.h};
            const OutView o[1] = {{dl, a.T, L.vc, L.vc}};
            typename EpiCeDlogits<float>::Params ep{lse_buf, a.targets, a.grad_scale, vvi, n_base};
            st = launch_gemm<float, 128, false, false, EpiCeDlogits<float>>("ce_bwd_logits_dl", A, B, o, nullptr, Ti, vci, hi,
                                                                            0, 0, n_base, 0, ep, s);
            if (st != TPCE_OK) return st;
        }
        if (a.dE) {
            if ((st = transpose_f32(dl, a.T, L.vc, L.vc, dlt, Tp, s)) != TPCE_OK) return st;
            Operand A{dlt, L.vc, a.T, Tp};  // K-major: M = vc rows, K = T columns
            Operand B{Ht, a.h, a.T, Tp};    // K-major: N = h rows, K = T columns
            const OutView o[1] = {{static_cast<float *>(a.dE) + static_cast<int64_t>(n_base) * a.h, L.vc, a.h, a.h}};
            st = launch_gemm<float, 128, false, false, EpiStore<float>>("ce_bwd_dE", A, B, o, nullptr, vci, hi, Ti, 0, 0, 0,
                                                                        0, {nullptr}, s);
            if (st != TPCE_OK) return st;
        }
        if (a.dH) {
            Operand A{dl, a.T, L.vc, L.vc};        // K-major [T, vc]
            Operand B{Et, a.h, a.v_pad, a.v_pad};  // K-major: N = h rows, K = v columns (from n_base)
            const OutView o[1] = {{a.dH, a.T, a.h, a.h}};
            st = launch_gemm<float, 128, false, false, EpiF32Accumulate>("ce_bwd_dH_shard_sum", A, B, o, nullptr, Ti, hi, vci,
                                                                         0, 0, 0, n_base, {c == 0 ? 0 : 1}, s);
            if (st != TPCE_OK) return st;
        }
    }
    return TPCE_OK;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_ce_workspace_bytes(int64_t T, int64_t h, int64_t v_pad, int t, int dtype, int with_grads) {
    if (check_ce_shape(T, h, v_pad, 1, t, dtype) != TPCE_OK) return 0;
    return ce_ws_layout(T, h, v_pad, t, with_grads != 0, dtype).total;
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
    const size_t esz = dtype == TPCE_F32 ? 4 : 2;
    if (T == 0) {
        if (dE && cudaMemsetAsync(dE, 0, static_cast<size_t>(v_pad) * h * esz, s) != cudaSuccess)
            return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const CeWs L = ce_ws_layout(T, h, v_pad, t, grads, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    float *lse_buf = lse ? lse : at<float>(ws, L.lse);
    const CeArgs a{H, E, targets, T, h, v_pad, v_valid, t, grad_scale, loss, lse, dH, dE};
    st = dtype == TPCE_F32 ? ce_forward<float>(a, L, ws, lse_buf, s) : ce_forward<__nv_bfloat16>(a, L, ws, lse_buf, s);
    if (st != TPCE_OK || !grads) return st;
    return dtype == TPCE_F32 ? ce_backward_f32(a, L, ws, lse_buf, s) : ce_backward_bf16(a, L, ws, lse_buf, s);
}
