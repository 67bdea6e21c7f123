// linear.cu -- the two linear primitives of Megatron's 1D tensor parallelism,
// ColumnParallelLinear and RowParallelLinear, with their t shards laid out on
// one GPU, and the attention projections built on them.
//
// "Distributed tensor parallelism: scale fine-tuning of 70B-parameter LLMs
// with Megatron-LM", sections "The Mechanics of Tensor Parallelism (TP) in
// Megatron-LM" and "The Multi-Head Attention Block"; "Mathematical
// Foundations of Megatron-LM 1D Slicing", sections "Column-Parallel Linear
// Layer", "Row-Parallel Linear Layer" and "Self-Attention Layer
// Decomposition".
//
// Both primitives compute Y = X W + b. They differ in the dimension of W the
// shards split, and so in where a shard sum falls:
//   column-parallel  W = [W_1 .. W_t] by columns. Forward: each shard's
//                    columns, no exchange. Backward: dX = sum_i dY_i W_i^T
//                    (f*), taken in the accumulator of the dX GEMM, whose K
//                    runs over the concatenated shard column ranges.
//   row-parallel     W = [W_1; ..; W_t] by rows, X by the matching columns.
//                    Forward: Y = sum_i X_i W_i (g) in the accumulator, then
//                    b once. Backward: each shard's columns of dX, no sum.
// On one GPU both are the same three GEMMs; the mode sets the validation and
// the kernel names.
//
// Sequence parallelism ("Mathematical Foundations ...", section "Sequence
// Parallelism"): the column-parallel entry reads the all-gathered X from t
// per-rank sequence chunks (and writes dX back into chunks); the
// row-parallel exit writes each shard-summed row of Y into the chunk that
// owns it (and reads the gathered dY from chunks in the backward).
//
// Attention: the fused QKV projection is column-parallel by heads (its
// columns grouped by key/value head, so that a contiguous split gives each
// shard whole heads: for each KV head g, the query heads sharing it, then K_g,
// then V_g); the output projection W_O is row-parallel over the concatenated
// head outputs. The attention core between them is not part of this library.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

constexpr int64_t kMaxDim = INT_MAX - 1024;  // kernel coordinates are 32-bit

struct LinearNames {
    const char *fwd, *dX, *dW;
};

tpce_status check_linear_shape(int64_t T, int64_t n_in, int64_t n_out, int t, int parallel, int dtype) {
    if (dtype != TPCE_BF16 && dtype != TPCE_F32) return TPCE_ERR_INVALID;
    if (parallel != TPCE_COLUMN_PARALLEL && parallel != TPCE_ROW_PARALLEL) return TPCE_ERR_INVALID;
    if (T < 0 || n_in < 8 || n_out < 8 || t < 1) return TPCE_ERR_SHAPE;
    if (T > kMaxDim || n_in > kMaxDim || n_out > kMaxDim) return TPCE_ERR_SHAPE;
    if (n_in % 8 != 0 || n_out % 8 != 0) return TPCE_ERR_SHAPE;  // 16-byte row pitch
    const int64_t split = parallel == TPCE_COLUMN_PARALLEL ? n_out : n_in;
    if (split % t != 0) return TPCE_ERR_SHAPE;         // equal shards
    if ((split / t) % 64 != 0) return TPCE_ERR_SHAPE;  // a shard is whole 64-wide blocks
    if (dtype == TPCE_F32 && (T + 31) / 32 > 65535) return TPCE_ERR_SHAPE;  // transpose grid
    return TPCE_OK;
}

inline int64_t pad4(int64_t x) { return (x + 3) / 4 * 4; }
inline int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }

// dW = X^T dY contracts over tokens with X's rows as its A operand, MN-major
// as X is stored: that costs the tensor core about 11% against a K-major A
// (measured on GB300). From an output width of 6144 on, X is first transposed
// into a K-major copy (4 T n_in bytes at HBM speed against 11% of 2 T n_in
// n_out FLOPs); with sequence-parallel X the copy is made chunk by chunk.
// bf16 calls only.
#ifndef TPCE_WGRAD_KMAJOR_MIN
#define TPCE_WGRAD_KMAJOR_MIN 6144
#endif
inline bool xt_copy(int64_t n_out, int dtype) { return dtype == TPCE_BF16 && n_out >= TPCE_WGRAD_KMAJOR_MIN; }

// Workspace: the column-sum partials (bias gradient), and where it pays the
// bf16 copy X^T [n_in, T] (rows padded to a multiple of 8); fp32 adds the
// transposed operands of the tf32 path: W^T (forward), X^T and dY^T (weight
// gradient), token-major ones with rows padded to a multiple of 4.
struct LinWs {
    size_t tail, partial, Wt, Xt, dYt, XtB, total;
};

LinWs lin_ws_layout(int64_t T, int64_t n_in, int64_t n_out, int dtype) {
    LinWs L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    L.tail = take(kTailScratchBytes);  // offset 0: all the bf16 forward needs
    L.partial = take(colsum_partial_floats(T, n_out) * sizeof(float));
    if (xt_copy(n_out, dtype)) L.XtB = take(static_cast<size_t>(n_in) * pad8(T) * 2);
    if (dtype == TPCE_F32) {
        const size_t Tp = static_cast<size_t>(pad4(T));
        L.Wt = take(static_cast<size_t>(n_out) * n_in * 4);
        L.Xt = take(static_cast<size_t>(n_in) * Tp * 4);
        L.dYt = take(static_cast<size_t>(n_out) * Tp * 4);
    }
    L.total = off;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// Sequence-chunked activations of one call (null members: dense tensors).
// Column-parallel entry: x (the X chunks) and out (dX chunks, backward).
// Row-parallel exit: out (the Y chunks, forward) and dy (dY chunks, backward).
struct LinSP {
    const Chunks *x;
    const Chunks *dy;
    const Chunks *out;
};

// Y = X W (+ b) on the bf16 path, with X or Y chunked as sp says.
template <typename ElemT>
tpce_status gemm_fwd(const char *name, const Operand &a, const Operand &bw, const OutView *o, int Ti, int oi, int ii,
                     const float *b, cudaStream_t s, const LinSP *sp, const TailScratch *ts) {
    constexpr bool kBf = std::is_same<ElemT, __nv_bfloat16>::value;
    if constexpr (kBf) {
        if (sp && sp->x)
            return launch_gemm_auto<ElemT, false, true, EpiStore<ElemT>, kBN192 | kBN256, kChunkA>(
                name, a, bw, o, nullptr, Ti, oi, ii, 0, 0, 0, 0, {b}, s, 0, sp->x, ts);
        if (sp && sp->out)
            return launch_gemm_auto<ElemT, false, true, EpiStore<ElemT>, kBN192 | kBN256, kChunkC>(
                name, a, bw, o, nullptr, Ti, oi, ii, 0, 0, 0, 0, {b}, s, 0, sp->out, ts);
        return launch_gemm_auto<ElemT, false, true, EpiStore<ElemT>, kBN192 | kBN256>(name, a, bw, o, nullptr, Ti, oi, ii,
                                                                                   0, 0, 0, 0, {b}, s, 0, nullptr, ts);
    } else {
        if (sp && sp->x)
            return launch_gemm<float, 128, false, false, EpiStore<float>, kChunkA>(name, a, bw, o, nullptr, Ti, oi, ii, 0,
                                                                                   0, 0, 0, {b}, s, true, 0, sp->x);
        if (sp && sp->out)
            return launch_gemm<float, 128, false, false, EpiStore<float>, kChunkC>(name, a, bw, o, nullptr, Ti, oi, ii, 0,
                                                                                   0, 0, 0, {b}, s, true, 0, sp->out);
        return launch_gemm<float, 128, false, false, EpiStore<float>>(name, a, bw, o, nullptr, Ti, oi, ii, 0, 0, 0, 0,
                                                                      {b}, s);
    }
}

// dX = dY W^T, with dY (row exit) or dX (column entry) chunked as sp says.
template <typename ElemT>
tpce_status gemm_dx(const char *name, const Operand &a, const Operand &bw, const OutView *o, int Ti, int ii, int oi,
                    cudaStream_t s, const LinSP *sp, const TailScratch *ts) {
    constexpr bool kBf = std::is_same<ElemT, __nv_bfloat16>::value;
    if constexpr (kBf) {
        if (sp && sp->dy)
            return launch_gemm_auto<ElemT, false, false, EpiStore<ElemT>, kBN192 | kBN256, kChunkA>(
                name, a, bw, o, nullptr, Ti, ii, oi, 0, 0, 0, 0, {nullptr}, s, 0, sp->dy, ts);
        if (sp && sp->out)
            return launch_gemm_auto<ElemT, false, false, EpiStore<ElemT>, kBN192 | kBN256, kChunkC>(
                name, a, bw, o, nullptr, Ti, ii, oi, 0, 0, 0, 0, {nullptr}, s, 0, sp->out, ts);
        return launch_gemm_auto<ElemT, false, false, EpiStore<ElemT>, kBN192 | kBN256>(name, a, bw, o, nullptr, Ti, ii,
                                                                                    oi, 0, 0, 0, 0, {nullptr}, s, 0,
                                                                                    nullptr, ts);
    } else {
        if (sp && sp->dy)
            return launch_gemm<float, 128, false, false, EpiStore<float>, kChunkA>(name, a, bw, o, nullptr, Ti, ii, oi, 0,
                                                                                   0, 0, 0, {nullptr}, s, true, 0, sp->dy);
        if (sp && sp->out)
            return launch_gemm<float, 128, false, false, EpiStore<float>, kChunkC>(
                name, a, bw, o, nullptr, Ti, ii, oi, 0, 0, 0, 0, {nullptr}, s, true, 0, sp->out);
        return launch_gemm<float, 128, false, false, EpiStore<float>>(name, a, bw, o, nullptr, Ti, ii, oi, 0, 0, 0, 0,
                                                                      {nullptr}, s);
    }
}

// The transpose of a [T, C] fp32 activation into out [C, Tp], from one buffer
// or from its sequence chunks (one column block of out per chunk).
tpce_status transpose_rows(const float *in, const Chunks *ch, int64_t T, int64_t C, float *out, int64_t Tp,
                           cudaStream_t s) {
    if (!ch) return transpose_f32(in, T, C, C, out, Tp, s);
    for (int c = 0; c < ch->count; ++c) {
        tpce_status st = transpose_f32(static_cast<const float *>(ch->ptrs[c]), ch->rows, C, C, out + c * ch->rows, Tp, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
}

tpce_status forward_impl(const LinearNames &nm, const void *X, const void *W, const float *b, int64_t T, int64_t n_in,
                         int64_t n_out, int dtype, void *Y, void *ws, const LinWs &L, cudaStream_t s,
                         const LinSP *sp, const TailScratch *ts) {
    const int Ti = static_cast<int>(T), ii = static_cast<int>(n_in), oi = static_cast<int>(n_out);
    const OutView o[1] = {{Y, T, n_out, n_out}};
    if (dtype == TPCE_BF16) {
        Operand a{X, T, n_in, n_in};      // K-major [T, n_in]
        Operand bw{W, n_in, n_out, n_out};  // MN-major: K = n_in rows, N = n_out columns
        return gemm_fwd<__nv_bfloat16>(nm.fwd, a, bw, o, Ti, oi, ii, b, s, sp, ts);
    }
    float *Wt = at<float>(ws, L.Wt);
    tpce_status st = transpose_f32(static_cast<const float *>(W), n_in, n_out, n_out, Wt, n_in, s);  // W^T
    if (st != TPCE_OK) return st;
    Operand a{X, T, n_in, n_in};       // K-major [T, n_in]
    Operand bw{Wt, n_out, n_in, n_in};  // K-major: N = n_out rows, K = n_in columns
    return gemm_fwd<float>(nm.fwd, a, bw, o, Ti, oi, ii, b, s, sp, nullptr);
}

tpce_status backward_impl(const LinearNames &nm, const void *dY, const void *X, const void *W, int64_t T, int64_t n_in,
                          int64_t n_out, int dtype, void *dX, void *dW, float *db, void *ws, const LinWs &L,
                          cudaStream_t s, const LinSP *sp) {
    const int Ti = static_cast<int>(T), ii = static_cast<int>(n_in), oi = static_cast<int>(n_out);
    float *partial = at<float>(ws, L.partial);
    const TailScratch tail{at<uint8_t>(ws, L.tail), kTailScratchBytes};
    const TailScratch *ts = &tail;
    tpce_status st;
    if (dtype == TPCE_BF16) {
        using bf = __nv_bfloat16;
        // dX = dY W^T (column-parallel: the f* sum over shards in the accumulator)
        {
            Operand a{dY, T, n_out, n_out};   // K-major [T, n_out]
            Operand bw{W, n_in, n_out, n_out};  // K-major: N = n_in rows, K = n_out columns
            const OutView o[1] = {{dX, T, n_in, n_in}};
            if ((st = gemm_dx<bf>(nm.dX, a, bw, o, Ti, ii, oi, s, sp, ts)) != TPCE_OK) return st;
        }
        // dW = X^T dY (each shard's own block of W)
        if (xt_copy(n_out, dtype)) {
            bf *Xt = at<bf>(ws, L.XtB);
            const int64_t Tp = pad8(T);
            if (sp && sp->x) {
                // the gathered X^T, one sequence chunk (a column block of X^T) at a time
                for (int c = 0; c < sp->x->count; ++c) {
                    st = transpose_bf16(sp->x->ptrs[c], sp->x->rows, n_in, n_in, Xt + c * sp->x->rows, Tp, s);
                    if (st != TPCE_OK) return st;
                }
            } else if ((st = transpose_bf16(X, T, n_in, n_in, Xt, Tp, s)) != TPCE_OK) {
                return st;
            }
            Operand a{Xt, n_in, T, Tp};       // K-major: M = n_in rows, K = T columns
            Operand bw{dY, T, n_out, n_out};  // MN-major: K = T rows, N = n_out columns (or the dY chunks)
            const OutView o[1] = {{dW, n_in, n_out, n_out}};
            st = (sp && sp->dy) ? launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256, kChunkB>(
                                      nm.dW, a, bw, o, nullptr, ii, oi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->dy, ts)
                                : launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>(
                                      nm.dW, a, bw, o, nullptr, ii, oi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, nullptr, ts);
            if (st != TPCE_OK) return st;
        } else {
            Operand a{X, T, n_in, n_in};     // MN-major: K = T rows, M = n_in columns
            Operand bw{dY, T, n_out, n_out};  // MN-major: K = T rows, N = n_out columns
            const OutView o[1] = {{dW, n_in, n_out, n_out}};
            if (sp && sp->x)
                st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256, kChunkA>(
                    nm.dW, a, bw, o, nullptr, ii, oi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->x, ts);
            else if (sp && sp->dy)
                st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256, kChunkB>(
                    nm.dW, a, bw, o, nullptr, ii, oi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->dy, ts);
            else
                st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>(nm.dW, a, bw, o, nullptr, ii, oi,
                                                                                      Ti, 0, 0, 0, 0, {nullptr}, s, 0,
                                                                                      nullptr, ts);
            if (st != TPCE_OK) return st;
        }
        if (db) {
            st = (sp && sp->dy) ? colsum_chunks(0, sp->dy->ptrs, sp->dy->count, sp->dy->rows, n_out, n_out, db,
                                                partial, s)
                                : colsum(0, dY, T, n_out, n_out, db, partial, s);
            if (st != TPCE_OK) return st;
        }
        return TPCE_OK;
    }
    const int64_t Tp = pad4(T);
    float *Xt = at<float>(ws, L.Xt), *dYt = at<float>(ws, L.dYt);
    {
        Operand a{dY, T, n_out, n_out};   // K-major [T, n_out]
        Operand bw{W, n_in, n_out, n_out};  // K-major: N = n_in rows, K = n_out columns
        const OutView o[1] = {{dX, T, n_in, n_in}};
        if ((st = gemm_dx<float>(nm.dX, a, bw, o, Ti, ii, oi, s, sp, nullptr)) != TPCE_OK) return st;
    }
    st = transpose_rows(static_cast<const float *>(X), sp ? sp->x : nullptr, T, n_in, Xt, Tp, s);
    if (st != TPCE_OK) return st;
    st = transpose_rows(static_cast<const float *>(dY), sp ? sp->dy : nullptr, T, n_out, dYt, Tp, s);
    if (st != TPCE_OK) return st;
    {
        Operand a{Xt, n_in, T, Tp};    // K-major: M = n_in rows, K = T columns
        Operand bw{dYt, n_out, T, Tp};  // K-major: N = n_out rows, K = T columns
        const OutView o[1] = {{dW, n_in, n_out, n_out}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>(nm.dW, a, bw, o, nullptr, ii, oi, Ti, 0, 0, 0, 0,
                                                                    {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    if (db) {
        st = (sp && sp->dy) ? colsum_chunks(1, sp->dy->ptrs, sp->dy->count, sp->dy->rows, n_out, n_out, db, partial, s)
                            : colsum(1, dY, T, n_out, n_out, db, partial, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
}

// With sp, the chunked activations are given there (already validated) and
// the matching dense pointers are unused.
tpce_status linear_forward(const LinearNames &nm, const void *X, const void *W, const float *b, int64_t T,
                           int64_t n_in, int64_t n_out, int t, int parallel, int dtype, void *Y, void *ws,
                           size_t ws_bytes, void *stream, const LinSP *sp = nullptr) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, parallel, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;  // no tokens: nothing to compute (token tensors may be NULL)
    if (!W || (!X && !(sp && sp->x)) || (!Y && !(sp && sp->out))) return TPCE_ERR_INVALID;
    for (const void *p : {X, W, static_cast<const void *>(b), static_cast<const void *>(Y),
                          static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    const LinWs L = lin_ws_layout(T, n_in, n_out, dtype);
    if (dtype == TPCE_F32 && (!ws || ws_bytes < L.total)) return TPCE_ERR_WORKSPACE;
    // the bf16 forward takes an optional workspace: its start splits the last wave's tiles
    const TailScratch tail = (ws && ws_bytes >= kTailScratchBytes) ? TailScratch{ws, kTailScratchBytes}
                                                                  : TailScratch{nullptr, 0};
    return forward_impl(nm, X, W, b, T, n_in, n_out, dtype, Y, ws, L, static_cast<cudaStream_t>(stream), sp, &tail);
}

tpce_status linear_backward(const LinearNames &nm, const void *dY, const void *X, const void *W, int64_t T,
                            int64_t n_in, int64_t n_out, int t, int parallel, int dtype, void *dX, void *dW, float *db,
                            void *ws, size_t ws_bytes, void *stream, const LinSP *sp = nullptr) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, parallel, dtype);
    if (st != TPCE_OK) return st;
    if (!W || !dW) return TPCE_ERR_INVALID;
    if (T > 0 && ((!dY && !(sp && sp->dy)) || (!X && !(sp && sp->x)) || (!dX && !(sp && sp->out))))
        return TPCE_ERR_INVALID;
    for (const void *p : {dY, X, W, static_cast<const void *>(dX), static_cast<const void *>(dW),
                          static_cast<const void *>(db), static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        // no tokens: the weight and bias gradients are empty sums
        const size_t esz = dtype == TPCE_F32 ? 4 : 2;
        if (cudaMemsetAsync(dW, 0, static_cast<size_t>(n_in) * n_out * esz, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (db && cudaMemsetAsync(db, 0, sizeof(float) * n_out, s) != cudaSuccess) return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const LinWs L = lin_ws_layout(T, n_in, n_out, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    return backward_impl(nm, dY, X, W, T, n_in, n_out, dtype, dX, dW, db, ws, L, s, sp);
}

// Sequence chunks of a [T, C] activation: t buffers of T/t rows (whole
// 128-row tile blocks), 16-byte aligned.
tpce_status check_chunks(const void *const *p, int64_t T, int t, Chunks &c) {
    if (!p) return TPCE_ERR_INVALID;
    if (t < 1 || t > kMaxChunks || T % t != 0 || (T / t) % 128 != 0) return TPCE_ERR_SHAPE;
    for (int i = 0; i < t; ++i) {
        if (!p[i]) return TPCE_ERR_INVALID;
        if (!aligned16(p[i])) return TPCE_ERR_ALIGN;
    }
    c = Chunks{p, T / t, t};
    return TPCE_OK;
}

// The sequence-parallel forms: the column-parallel entry (X chunks in; dX
// chunks out of the backward) and the row-parallel exit (Y chunks out; dY
// chunks into the backward).
tpce_status column_forward_sp(const LinearNames &nm, const void *const *X_chunks, const void *W, const float *b,
                              int64_t T, int64_t n_in, int64_t n_out, int t, int dtype, void *Y, void *ws,
                              size_t ws_bytes, void *stream) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, TPCE_COLUMN_PARALLEL, dtype);
    if (st != TPCE_OK || T == 0) return st;
    Chunks xc{};
    if ((st = check_chunks(X_chunks, T, t, xc)) != TPCE_OK) return st;
    const LinSP sp{&xc, nullptr, nullptr};
    return linear_forward(nm, nullptr, W, b, T, n_in, n_out, t, TPCE_COLUMN_PARALLEL, dtype, Y, ws, ws_bytes, stream,
                          &sp);
}

tpce_status column_backward_sp(const LinearNames &nm, const void *dY, const void *const *X_chunks, const void *W,
                               int64_t T, int64_t n_in, int64_t n_out, int t, int dtype, void *const *dX_chunks,
                               void *dW, float *db, void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, TPCE_COLUMN_PARALLEL, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0)
        return linear_backward(nm, nullptr, nullptr, W, 0, n_in, n_out, t, TPCE_COLUMN_PARALLEL, dtype, nullptr, dW, db,
                               ws, ws_bytes, stream);
    Chunks xc{}, dxc{};
    if ((st = check_chunks(X_chunks, T, t, xc)) != TPCE_OK) return st;
    if ((st = check_chunks(reinterpret_cast<const void *const *>(dX_chunks), T, t, dxc)) != TPCE_OK) return st;
    const LinSP sp{&xc, nullptr, &dxc};
    return linear_backward(nm, dY, nullptr, W, T, n_in, n_out, t, TPCE_COLUMN_PARALLEL, dtype, nullptr, dW, db, ws,
                           ws_bytes, stream, &sp);
}

tpce_status row_forward_sp(const LinearNames &nm, const void *X, const void *W, const float *b, int64_t T, int64_t n_in,
                           int64_t n_out, int t, int dtype, void *const *Y_chunks, void *ws, size_t ws_bytes,
                           void *stream) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, TPCE_ROW_PARALLEL, dtype);
    if (st != TPCE_OK || T == 0) return st;
    Chunks yc{};
    if ((st = check_chunks(reinterpret_cast<const void *const *>(Y_chunks), T, t, yc)) != TPCE_OK) return st;
    const LinSP sp{nullptr, nullptr, &yc};
    return linear_forward(nm, X, W, b, T, n_in, n_out, t, TPCE_ROW_PARALLEL, dtype, nullptr, ws, ws_bytes, stream, &sp);
}

tpce_status row_backward_sp(const LinearNames &nm, const void *const *dY_chunks, const void *X, const void *W,
                            int64_t T, int64_t n_in, int64_t n_out, int t, int dtype, void *dX, void *dW, float *db,
                            void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_linear_shape(T, n_in, n_out, t, TPCE_ROW_PARALLEL, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0)
        return linear_backward(nm, nullptr, nullptr, W, 0, n_in, n_out, t, TPCE_ROW_PARALLEL, dtype, nullptr, dW, db,
                               ws, ws_bytes, stream);
    Chunks dyc{};
    if ((st = check_chunks(dY_chunks, T, t, dyc)) != TPCE_OK) return st;
    const LinSP sp{nullptr, &dyc, nullptr};
    return linear_backward(nm, nullptr, X, W, T, n_in, n_out, t, TPCE_ROW_PARALLEL, dtype, dX, dW, db, ws, ws_bytes,
                           stream, &sp);
}

const LinearNames kColumnNames{"linear_column_fwd", "linear_column_bwd_dX_shard_sum", "linear_column_bwd_dW"};
const LinearNames kRowNames{"linear_row_fwd_shard_sum", "linear_row_bwd_dX", "linear_row_bwd_dW"};
const LinearNames kQkvNames{"attn_qkv_fwd", "attn_qkv_bwd_dX_shard_sum", "attn_qkv_bwd_dW"};
const LinearNames kOutNames{"attn_out_fwd_shard_sum", "attn_out_bwd_dO", "attn_out_bwd_dW"};

inline const LinearNames &linear_names(int parallel) {
    return parallel == TPCE_ROW_PARALLEL ? kRowNames : kColumnNames;
}

// Head counts of the attention projections: whole key/value groups per shard.
tpce_status check_heads(int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, int t) {
    if (n_heads < 1 || n_kv_heads < 1 || head_dim < 8 || t < 1) return TPCE_ERR_SHAPE;
    if (n_heads % n_kv_heads != 0) return TPCE_ERR_SHAPE;  // query heads share key/value heads evenly
    if (n_kv_heads % t != 0) return TPCE_ERR_SHAPE;        // each shard holds whole key/value heads
    if (head_dim % 8 != 0) return TPCE_ERR_SHAPE;
    if (n_heads + 2 * n_kv_heads > kMaxDim / head_dim) return TPCE_ERR_SHAPE;
    return TPCE_OK;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_linear_workspace_bytes(int64_t T, int64_t n_in, int64_t n_out, int t, int parallel,
                                              int dtype) {
    if (check_linear_shape(T, n_in, n_out, t, parallel, dtype) != TPCE_OK) return 0;
    return lin_ws_layout(T, n_in, n_out, dtype).total;
}

extern "C" tpce_status tp_linear_forward(const void *X, const void *W, const float *b, int64_t T, int64_t n_in,
                                         int64_t n_out, int t, int parallel, int dtype, void *Y, void *ws,
                                         size_t ws_bytes, void *stream) {
    return linear_forward(linear_names(parallel), X, W, b, T, n_in, n_out, t, parallel, dtype, Y, ws, ws_bytes,
                          stream);
}

extern "C" tpce_status tp_linear_backward(const void *dY, const void *X, const void *W, int64_t T, int64_t n_in,
                                          int64_t n_out, int t, int parallel, int dtype, void *dX, void *dW, float *db,
                                          void *ws, size_t ws_bytes, void *stream) {
    return linear_backward(linear_names(parallel), dY, X, W, T, n_in, n_out, t, parallel, dtype, dX, dW, db, ws,
                           ws_bytes, stream);
}

extern "C" size_t tpce_attn_workspace_bytes(int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                            int64_t head_dim, int t, int dtype) {
    if (check_heads(n_heads, n_kv_heads, head_dim, t) != TPCE_OK) return 0;
    const int64_t qkv = (n_heads + 2 * n_kv_heads) * head_dim, hq = n_heads * head_dim;
    const size_t a = tpce_linear_workspace_bytes(T, h, qkv, t, TPCE_COLUMN_PARALLEL, dtype);
    const size_t b = tpce_linear_workspace_bytes(T, hq, h, t, TPCE_ROW_PARALLEL, dtype);
    if (a == 0 || b == 0) return 0;
    return a > b ? a : b;
}

extern "C" tpce_status tp_attn_qkv_forward(const void *X, const void *Wqkv, const float *bqkv, int64_t T, int64_t h,
                                           int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, int t, int dtype,
                                           void *QKV, void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_heads(n_heads, n_kv_heads, head_dim, t);
    if (st != TPCE_OK) return st;
    return linear_forward(kQkvNames, X, Wqkv, bqkv, T, h, (n_heads + 2 * n_kv_heads) * head_dim, t,
                          TPCE_COLUMN_PARALLEL, dtype, QKV, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_qkv_backward(const void *dQKV, const void *X, const void *Wqkv, int64_t T, int64_t h,
                                            int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, int t, int dtype,
                                            void *dX, void *dWqkv, float *dbqkv, void *ws, size_t ws_bytes,
                                            void *stream) {
    tpce_status st = check_heads(n_heads, n_kv_heads, head_dim, t);
    if (st != TPCE_OK) return st;
    return linear_backward(kQkvNames, dQKV, X, Wqkv, T, h, (n_heads + 2 * n_kv_heads) * head_dim, t,
                           TPCE_COLUMN_PARALLEL, dtype, dX, dWqkv, dbqkv, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_out_forward(const void *O, const void *Wo, const float *bo, int64_t T, int64_t h,
                                           int64_t n_heads, int64_t head_dim, int t, int dtype, void *Z, void *ws,
                                           size_t ws_bytes, void *stream) {
    if (n_heads < 1 || head_dim < 8 || head_dim % 8 != 0 || n_heads % t != 0 || n_heads > kMaxDim / head_dim)
        return TPCE_ERR_SHAPE;
    return linear_forward(kOutNames, O, Wo, bo, T, n_heads * head_dim, h, t, TPCE_ROW_PARALLEL, dtype, Z, ws, ws_bytes,
                          stream);
}

extern "C" tpce_status tp_attn_out_backward(const void *dZ, const void *O, const void *Wo, int64_t T, int64_t h,
                                            int64_t n_heads, int64_t head_dim, int t, int dtype, void *dO, void *dWo,
                                            float *dbo, void *ws, size_t ws_bytes, void *stream) {
    if (n_heads < 1 || head_dim < 8 || head_dim % 8 != 0 || n_heads % t != 0 || n_heads > kMaxDim / head_dim)
        return TPCE_ERR_SHAPE;
    return linear_backward(kOutNames, dZ, O, Wo, T, n_heads * head_dim, h, t, TPCE_ROW_PARALLEL, dtype, dO, dWo, dbo,
                           ws, ws_bytes, stream);
}

extern "C" tpce_status tp_column_linear_forward_sp(const void *const *X_chunks, const void *W, const float *b,
                                                   int64_t T, int64_t n_in, int64_t n_out, int t, int dtype, void *Y,
                                                   void *ws, size_t ws_bytes, void *stream) {
    return column_forward_sp(kColumnNames, X_chunks, W, b, T, n_in, n_out, t, dtype, Y, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_column_linear_backward_sp(const void *dY, const void *const *X_chunks, const void *W,
                                                    int64_t T, int64_t n_in, int64_t n_out, int t, int dtype,
                                                    void *const *dX_chunks, void *dW, float *db, void *ws,
                                                    size_t ws_bytes, void *stream) {
    return column_backward_sp(kColumnNames, dY, X_chunks, W, T, n_in, n_out, t, dtype, dX_chunks, dW, db, ws, ws_bytes,
                              stream);
}

extern "C" tpce_status tp_row_linear_forward_sp(const void *X, const void *W, const float *b, int64_t T, int64_t n_in,
                                                int64_t n_out, int t, int dtype, void *const *Y_chunks, void *ws,
                                                size_t ws_bytes, void *stream) {
    return row_forward_sp(kRowNames, X, W, b, T, n_in, n_out, t, dtype, Y_chunks, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_row_linear_backward_sp(const void *const *dY_chunks, const void *X, const void *W, int64_t T,
                                                 int64_t n_in, int64_t n_out, int t, int dtype, void *dX, void *dW,
                                                 float *db, void *ws, size_t ws_bytes, void *stream) {
    return row_backward_sp(kRowNames, dY_chunks, X, W, T, n_in, n_out, t, dtype, dX, dW, db, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_qkv_forward_sp(const void *const *X_chunks, const void *Wqkv, const float *bqkv,
                                              int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                              int64_t head_dim, int t, int dtype, void *QKV, void *ws, size_t ws_bytes,
                                              void *stream) {
    tpce_status st = check_heads(n_heads, n_kv_heads, head_dim, t);
    if (st != TPCE_OK) return st;
    return column_forward_sp(kQkvNames, X_chunks, Wqkv, bqkv, T, h, (n_heads + 2 * n_kv_heads) * head_dim, t, dtype,
                             QKV, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_qkv_backward_sp(const void *dQKV, const void *const *X_chunks, const void *Wqkv,
                                               int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                               int64_t head_dim, int t, int dtype, void *const *dX_chunks,
                                               void *dWqkv, float *dbqkv, void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_heads(n_heads, n_kv_heads, head_dim, t);
    if (st != TPCE_OK) return st;
    return column_backward_sp(kQkvNames, dQKV, X_chunks, Wqkv, T, h, (n_heads + 2 * n_kv_heads) * head_dim, t, dtype,
                              dX_chunks, dWqkv, dbqkv, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_out_forward_sp(const void *O, const void *Wo, const float *bo, int64_t T, int64_t h,
                                              int64_t n_heads, int64_t head_dim, int t, int dtype,
                                              void *const *Z_chunks, void *ws, size_t ws_bytes, void *stream) {
    if (n_heads < 1 || head_dim < 8 || head_dim % 8 != 0 || n_heads % t != 0 || n_heads > kMaxDim / head_dim)
        return TPCE_ERR_SHAPE;
    return row_forward_sp(kOutNames, O, Wo, bo, T, n_heads * head_dim, h, t, dtype, Z_chunks, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_attn_out_backward_sp(const void *const *dZ_chunks, const void *O, const void *Wo, int64_t T,
                                               int64_t h, int64_t n_heads, int64_t head_dim, int t, int dtype,
                                               void *dO, void *dWo, float *dbo, void *ws, size_t ws_bytes,
                                               void *stream) {
    if (n_heads < 1 || head_dim < 8 || head_dim % 8 != 0 || n_heads % t != 0 || n_heads > kMaxDim / head_dim)
        return TPCE_ERR_SHAPE;
    return row_backward_sp(kOutNames, dZ_chunks, O, Wo, T, n_heads * head_dim, h, t, dtype, dO, dWo, dbo, ws, ws_bytes,
                           stream);
}
