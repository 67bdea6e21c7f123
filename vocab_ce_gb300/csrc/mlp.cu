// mlp.cu -- the Megatron 1D tensor-parallel MLP block with its t shards laid
// out on one GPU: tp_mlp_forward / tp_mlp_backward (GeLU) and
// tp_swiglu_forward / tp_swiglu_backward (the SwiGLU variant).
//
// GeLU block ("Mathematical Foundations of Megatron-LM 1D Slicing", sections
// "Column-Parallel Linear Layer" and "Row-Parallel Linear Layer"):
//   GEMM1  U = X A + bA, Y = GeLU(U)  -- N runs over the concatenated column
//          blocks A_1..A_t; GeLU is applied in the epilogue, per shard, with
//          no exchange (it is elementwise).
//   GEMM2  Z = sum_i Y_i B_i + bB     -- K runs over the concatenated row
//          blocks B_1..B_t, so the accumulator sums the shard partials Z_i:
//          the forward operator g. bB is added once, in the epilogue.
// Backward (same page, "Conjugate Communication Operators"): g* hands dZ to
// every shard; f* sums the shard partials of dX, again in the accumulator of
// the dX GEMM (K over the concatenated shard ranges).
//
// SwiGLU block ("Distributed tensor parallelism: scale fine-tuning of
// 70B-parameter LLMs with Megatron-LM", section "The MLP Block"):
// Y = Swish(X W_gate) (.) (X W_up), Z = Y W_down. W1 = [W_gate | W_up] is one
// [h, 2f] matrix; shard i owns gate columns i f/t.. and the same up columns.
// GEMM1 runs on gated tiles: each accumulator holds the gate and the up
// columns of the same output columns, so Swish(G) Up is formed in the
// epilogue. GEMM2 and the g / f* shard sums are the GeLU block's; the
// backward's dY epilogue forms [dG | dUp] and the weight-gradient and dX
// GEMMs run over the 2f columns of W1.
//
// Sequence-parallel form ([MF] "Sequence Parallelism"): X, Z, dZ and dX may
// come as t sequence chunks in t buffers, one per rank. GEMM1 (and the dA
// GEMM) then read the all-gathered X straight from the chunks; GEMM2's (and
// the dX GEMM's) epilogue writes each tile's shard-summed rows into the chunk
// that owns them -- the reduce-scatter exit; the backward reads the
// all-gathered dZ from its chunks.
//
// bf16 tensors use the bf16 tensor-core path with operands read in place in
// either major order, except the A operands of the weight gradients at large
// widths (X^T, Y^T copies, below). fp32 tensors use the tf32 path, whose operands are
// K-major: the operands stored the other way (the weights in the forward; Y,
// dZ, X and the pre-activation gradient in the weight gradients) are first
// transposed into the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

constexpr int64_t kMaxDim = INT_MAX - 1024;  // kernel coordinates are 32-bit

// The nonlinearity between the two GEMMs.
enum class Act { GeLU, SwiGLU };

// Columns of the first GEMM's output (and of W1, b1, dU): f, or 2f for SwiGLU.
inline int64_t pre_width(Act act, int64_t f) { return act == Act::SwiGLU ? 2 * f : f; }

tpce_status check_mlp_shape(Act act, int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (dtype != TPCE_BF16 && dtype != TPCE_F32) return TPCE_ERR_INVALID;
    if (T < 0 || h < 8 || f < 1 || t < 1) return TPCE_ERR_SHAPE;
    if (T > kMaxDim || h > kMaxDim || pre_width(act, f) > kMaxDim) return TPCE_ERR_SHAPE;
    if (h % 8 != 0) return TPCE_ERR_SHAPE;           // 16-byte row pitch
    if (f % t != 0) return TPCE_ERR_SHAPE;           // equal shards
    if ((f / t) % 64 != 0) return TPCE_ERR_SHAPE;    // a shard is whole 64-wide blocks
    if (dtype == TPCE_F32 && (T + 31) / 32 > 65535) return TPCE_ERR_SHAPE;  // transpose grid
    return TPCE_OK;
}

inline int64_t pad4(int64_t x) { return (x + 3) / 4 * 4; }  // fp32 rows padded to 16 bytes
inline int64_t pad8(int64_t x) { return (x + 7) / 8 * 8; }  // bf16 rows padded to 16 bytes

// The weight gradients dB = Y^T dZ and dA = X^T dU contract over tokens, and
// with Y and X stored token-major their A operand is MN-major, which costs the
// tensor core about 11% against a K-major A (measured on GB300). A transposed
// copy (an HBM-bound pass of 4 T n bytes for an [T, n] operand) pays when the
// GEMM's other width is large: dA = X^T dU does 2 T h fw FLOPs over X's
// 4 T h bytes, dB = Y^T dZ 2 T f h over Y's 4 T f bytes, and the copy wins for
// that other width above about 4,500 on GB300. bf16 only; the
// sequence-parallel forms transpose X chunk by chunk into the column blocks of
// one X^T, and keep reading dZ (the B operand) from its chunks.
#ifndef TPCE_WGRAD_KMAJOR_MIN
#define TPCE_WGRAD_KMAJOR_MIN 6144
#endif
inline bool xt_copy(int64_t fw, int dtype) { return dtype == TPCE_BF16 && fw >= TPCE_WGRAD_KMAJOR_MIN; }
inline bool yt_copy(int64_t h, int dtype) { return dtype == TPCE_BF16 && h >= TPCE_WGRAD_KMAJOR_MIN; }

// Sequence-chunked activations (null members: dense tensors).
struct SeqPar {
    const Chunks *x;    // the X chunks: A of GEMM1 and of dA
    const Chunks *dz;   // the dZ chunks: A of dY, B of dB, the dbB column sum
    const Chunks *out;  // the Z chunks (forward) or dX chunks (backward): output map 0
};

// The split-tail scratch at the start of a workspace of at least ws_bytes
// (null when the workspace is missing or too small: tails run unsplit).
inline TailScratch tail_of(void *ws, size_t ws_bytes) {
    return (ws && ws_bytes >= kTailScratchBytes) ? TailScratch{ws, kTailScratchBytes} : TailScratch{nullptr, 0};
}

// Workspace layout. bf16: dU [T, fw] (fw = f, or 2f for SwiGLU: [dG | dUp]),
// the column-sum partials, and where they pay the transposed copies X^T
// [h, T] and Y^T [f, T] (rows padded to a multiple of 8) for K-major weight
// gradients. fp32 adds the transposed operands of the tf32 path: W1^T, W2^T
// (forward), Y^T, dZ^T, X^T, dU^T (backward), the token-major ones with rows
// padded to a multiple of 4.
struct MlpWs {
    size_t tail, dU, partial, At, Bt, Yt, dZt, Xt, dUt, XtB, YtB, total;
};

MlpWs mlp_ws_layout(Act act, int64_t T, int64_t h, int64_t f, int dtype) {
    MlpWs L{};
    const size_t esz = dtype == TPCE_F32 ? 4 : 2;
    const int64_t fw = pre_width(act, f);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    L.tail = take(kTailScratchBytes);  // offset 0: all the bf16 forward needs
    L.dU = take(static_cast<size_t>(T) * fw * esz);
    const size_t pf = std::max(colsum_partial_floats(T, fw), colsum_partial_floats(T, h));
    L.partial = take(pf * sizeof(float));
    if (xt_copy(fw, dtype)) L.XtB = take(static_cast<size_t>(h) * pad8(T) * 2);
    if (yt_copy(h, dtype)) L.YtB = take(static_cast<size_t>(f) * pad8(T) * 2);
    if (dtype == TPCE_F32) {
        const size_t Tp = static_cast<size_t>(pad4(T));
        L.At = take(static_cast<size_t>(fw) * h * 4);
        L.Bt = take(static_cast<size_t>(h) * f * 4);
        L.Yt = take(static_cast<size_t>(f) * Tp * 4);
        L.dZt = take(static_cast<size_t>(h) * Tp * 4);
        L.Xt = take(static_cast<size_t>(h) * Tp * 4);
        L.dUt = take(static_cast<size_t>(fw) * Tp * 4);
    }
    L.total = off;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// ---------------------------------------------------------------- bf16 path
// Forward. GeLU: A [h, f], U_save = U [T, f]. SwiGLU: A = W1 [h, 2f],
// U_save = [G | Up] [T, 2f].
tpce_status forward_bf16(Act act, const void *X, const void *A, const float *bA, const void *B, const float *bB,
                         int64_t T, int64_t h, int64_t f, void *Z, void *U, void *Y, cudaStream_t s,
                         const SeqPar *sp, const TailScratch *ts) {
    using bf = __nv_bfloat16;
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    const int64_t fw = pre_width(act, f);
    tpce_status st;
    Operand a{X, T, h, h};    // K-major [T, h]
    Operand b{A, h, fw, fw};  // MN-major: K = h rows, N = fw columns
    const OutView o1[2] = {{U, T, fw, fw}, {Y, T, f, f}};
    if (act == Act::GeLU) {
        // GEMM1 (column-parallel): U = X A + bA, Y = GeLU(U)
        st = sp ? launch_gemm_auto<bf, false, true, EpiBiasGelu<bf>, kBN192 | kBN256, kChunkA>(
                      "mlp_fwd_gemm1_bias_gelu", a, b, o1, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA}, s, 0, sp->x, ts)
                : launch_gemm_auto<bf, false, true, EpiBiasGelu<bf>, kBN192 | kBN256>(
                      "mlp_fwd_gemm1_bias_gelu", a, b, o1, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA}, s, 0, nullptr, ts);
    } else {
        // GEMM1 (column-parallel, gated): [G | Up] = X W1 + b1, Y = Swish(G) Up
        st = sp ? launch_gemm_auto<bf, false, true, EpiSwiGlu<bf>, kBN128 | kBN256, kChunkA>(
                      "swiglu_fwd_gemm1_gate_up", a, b, o1, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA, fi}, s, fi, sp->x, ts)
                : launch_gemm_auto<bf, false, true, EpiSwiGlu<bf>, kBN128 | kBN256>(
                      "swiglu_fwd_gemm1_gate_up", a, b, o1, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA, fi}, s, fi, nullptr,
                      ts);
    }
    if (st != TPCE_OK) return st;
    // GEMM2 (row-parallel) + g: Z = sum_i Y_i B_i + bB (sequence-parallel:
    // each row of Z into the chunk of its rank, the reduce-scatter exit)
    Operand a2{Y, T, f, f};  // K-major [T, f]
    Operand b2{B, f, h, h};  // MN-major: K = f rows, N = h columns
    const OutView o2[1] = {{Z, T, h, h}};
    const char *n2 = act == Act::GeLU ? "mlp_fwd_gemm2_shard_sum" : "swiglu_fwd_gemm2_shard_sum";
    if (sp)
        return launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256, kChunkC>(
            n2, a2, b2, o2, nullptr, Ti, hi, fi, 0, 0, 0, 0, {bB}, s, 0, sp->out, ts);
    return launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>(n2, a2, b2, o2, nullptr, Ti, hi, fi, 0, 0,
                                                                             0, 0, {bB}, s, 0, nullptr, ts);
}

tpce_status backward_bf16(Act act, const void *dZ, const void *X, const void *A, const void *B, const void *U,
                          const void *Y, int64_t T, int64_t h, int64_t f, void *dX, void *dA, float *dbA, void *dB,
                          float *dbB, void *ws, const MlpWs &L, cudaStream_t s, const SeqPar *sp) {
    using bf = __nv_bfloat16;
    const TailScratch tail{at<uint8_t>(ws, L.tail), kTailScratchBytes};
    const TailScratch *ts = &tail;
    bf *dU = at<bf>(ws, L.dU);
    float *partial = at<float>(ws, L.partial);
    const int64_t fw = pre_width(act, f);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f),
              fwi = static_cast<int>(fw);
    const bool glu = act == Act::SwiGLU;
    tpce_status st;
    // g* is the identity: every shard reads the same dZ.
    // dY_i = dZ B_i^T, fused with dU_i = dY_i (.) GeLU'(U_i), or for SwiGLU
    // with [dG_i | dUp_i] from the saved [G_i | Up_i]
    {
        Operand a{dZ, T, h, h};  // K-major [T, h]
        Operand b{B, f, h, h};   // K-major: N = f rows, K = h columns
        const OutView o[1] = {{dU, T, fw, fw}};
        const OutView in[1] = {{const_cast<void *>(U), T, fw, fw}};  // read by TMA, never written
        if (!glu)
            st = sp ? launch_gemm_auto<bf, false, false, EpiGeluGrad<bf>, kBN192 | kBN256, kChunkA>(
                          "mlp_bwd_dY_gelu_grad", a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {}, s, 0, sp->dz, ts)
                    : launch_gemm_auto<bf, false, false, EpiGeluGrad<bf>, kBN192 | kBN256>(
                          "mlp_bwd_dY_gelu_grad", a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {}, s, 0, nullptr, ts);
        else
            st = sp ? launch_gemm_auto<bf, false, false, EpiSwiGluGrad<bf>, kBN192 | kBN256, kChunkA>(
                          "swiglu_bwd_dY_swiglu_grad", a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {fi}, s, 0, sp->dz, ts)
                    : launch_gemm_auto<bf, false, false, EpiSwiGluGrad<bf>, kBN192 | kBN256>(
                          "swiglu_bwd_dY_swiglu_grad", a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {fi}, s, 0, nullptr, ts);
        if (st != TPCE_OK) return st;
    }
    const int64_t Tp = pad8(T);
    // dB_i = Y_i^T dZ
    {
        const char *nm = glu ? "swiglu_bwd_dW2" : "mlp_bwd_dB";
        Operand b{dZ, T, h, h};  // MN-major: K = T rows, N = h columns
        const OutView o[1] = {{dB, f, h, h}};
        if (yt_copy(h, TPCE_BF16)) {
            bf *Yt = at<bf>(ws, L.YtB);
            if ((st = transpose_bf16(Y, T, f, f, Yt, Tp, s)) != TPCE_OK) return st;
            Operand a{Yt, f, T, Tp};  // K-major: M = f rows, K = T columns
            st = sp ? launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256, kChunkB>(
                          nm, a, b, o, nullptr, fi, hi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->dz, ts)
                    : launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>(
                          nm, a, b, o, nullptr, fi, hi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, nullptr, ts);
        } else {
            Operand a{Y, T, f, f};  // MN-major: K = T rows, M = f columns
            st = sp ? launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256, kChunkB>(
                          nm, a, b, o, nullptr, fi, hi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->dz, ts)
                    : launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>(
                          nm, a, b, o, nullptr, fi, hi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, nullptr, ts);
        }
        if (st != TPCE_OK) return st;
    }
    // dA_i = X^T dU_i
    {
        const char *nm = glu ? "swiglu_bwd_dW1" : "mlp_bwd_dA";
        Operand b{dU, T, fw, fw};  // MN-major: K = T rows, N = fw columns
        const OutView o[1] = {{dA, h, fw, fw}};
        if (xt_copy(fw, TPCE_BF16)) {
            bf *Xt = at<bf>(ws, L.XtB);
            if (sp) {
                // the gathered X^T, one sequence chunk (a column block of X^T) at a time
                for (int c = 0; c < sp->x->count; ++c) {
                    const int64_t r0 = c * sp->x->rows;
                    st = transpose_bf16(sp->x->ptrs[c], sp->x->rows, h, h, Xt + r0, Tp, s);
                    if (st != TPCE_OK) return st;
                }
            } else if ((st = transpose_bf16(X, T, h, h, Xt, Tp, s)) != TPCE_OK) {
                return st;
            }
            Operand a{Xt, h, T, Tp};  // K-major: M = h rows, K = T columns
            st = launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>(nm, a, b, o, nullptr, hi, fwi, Ti, 0,
                                                                                   0, 0, 0, {nullptr}, s, 0, nullptr, ts);
        } else {
            Operand a{X, T, h, h};  // MN-major: K = T rows, M = h columns
            st = sp ? launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256, kChunkA>(
                          nm, a, b, o, nullptr, hi, fwi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, sp->x, ts)
                    : launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>(
                          nm, a, b, o, nullptr, hi, fwi, Ti, 0, 0, 0, 0, {nullptr}, s, 0, nullptr, ts);
        }
        if (st != TPCE_OK) return st;
    }
    // f*: dX = sum_i dU_i A_i^T, the shard sum taken in the accumulator
    {
        Operand a{dU, T, fw, fw};  // K-major [T, fw]
        Operand b{A, h, fw, fw};   // K-major: N = h rows, K = fw columns
        const OutView o[1] = {{dX, T, h, h}};
        const char *nm = glu ? "swiglu_bwd_dX_shard_sum" : "mlp_bwd_dX_shard_sum";
        st = sp ? launch_gemm_auto<bf, false, false, EpiStore<bf>, kBN192 | kBN256, kChunkC>(
                      nm, a, b, o, nullptr, Ti, hi, fwi, 0, 0, 0, 0, {nullptr}, s, 0, sp->out, ts)
                : launch_gemm_auto<bf, false, false, EpiStore<bf>, kBN192 | kBN256>(nm, a, b, o, nullptr, Ti, hi, fwi, 0,
                                                                                     0, 0, 0, {nullptr}, s, 0, nullptr,
                                                                                     ts);
        if (st != TPCE_OK) return st;
    }
    if (dbA && (st = colsum(0, dU, T, fw, fw, dbA, partial, s)) != TPCE_OK) return st;
    if (dbB) {
        st = sp ? colsum_chunks(0, sp->dz->ptrs, sp->dz->count, sp->dz->rows, h, h, dbB, partial, s)
                : colsum(0, dZ, T, h, h, dbB, partial, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
}

// ---------------------------------------------------------------- fp32 (tf32) path
tpce_status forward_f32(Act act, const float *X, const float *A, const float *bA, const float *B, const float *bB,
                        int64_t T, int64_t h, int64_t f, float *Z, float *U, float *Y, void *ws, const MlpWs &L,
                        cudaStream_t s, const SeqPar *sp) {
    float *At = at<float>(ws, L.At), *Bt = at<float>(ws, L.Bt);
    const int64_t fw = pre_width(act, f);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    tpce_status st = transpose_f32(A, h, fw, fw, At, h, s);  // A^T [fw, h]
    if (st != TPCE_OK) return st;
    if ((st = transpose_f32(B, f, h, h, Bt, f, s)) != TPCE_OK) return st;  // B^T [h, f]
    {
        Operand a{X, T, h, h};    // K-major [T, h]
        Operand b{At, fw, h, h};  // K-major: N = fw rows, K = h columns
        const OutView o[2] = {{U, T, fw, fw}, {Y, T, f, f}};
        const char *nm = act == Act::GeLU ? "mlp_fwd_gemm1_bias_gelu" : "swiglu_fwd_gemm1_gate_up";
        if (act == Act::GeLU)
            st = sp ? launch_gemm<float, 128, false, false, EpiBiasGelu<float>, kChunkA>(
                          nm, a, b, o, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA}, s, true, 0, sp->x)
                    : launch_gemm<float, 128, false, false, EpiBiasGelu<float>>(nm, a, b, o, nullptr, Ti, fi, hi, 0, 0,
                                                                                0, 0, {bA}, s);
        else  // gated tiles: rows n.. of W1^T are gate columns, rows f + n.. the up columns
            st = sp ? launch_gemm<float, 128, false, false, EpiSwiGlu<float>, kChunkA>(
                          nm, a, b, o, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA, fi}, s, true, fi, sp->x)
                    : launch_gemm<float, 128, false, false, EpiSwiGlu<float>>(nm, a, b, o, nullptr, Ti, fi, hi, 0, 0, 0,
                                                                              0, {bA, fi}, s, true, fi);
        if (st != TPCE_OK) return st;
    }
    Operand a2{Y, T, f, f};   // K-major [T, f]
    Operand b2{Bt, h, f, f};  // K-major: N = h rows, K = f columns
    const OutView o2[1] = {{Z, T, h, h}};
    const char *n2 = act == Act::GeLU ? "mlp_fwd_gemm2_shard_sum" : "swiglu_fwd_gemm2_shard_sum";
    if (sp)
        return launch_gemm<float, 128, false, false, EpiStore<float>, kChunkC>(n2, a2, b2, o2, nullptr, Ti, hi, fi, 0, 0,
                                                                               0, 0, {bB}, s, true, 0, sp->out);
    return launch_gemm<float, 128, false, false, EpiStore<float>>(n2, a2, b2, o2, nullptr, Ti, hi, fi, 0, 0, 0, 0, {bB},
                                                                  s);
}

tpce_status backward_f32(Act act, const float *dZ, const float *X, const float *A, const float *B, const float *U,
                         const float *Y, int64_t T, int64_t h, int64_t f, float *dX, float *dA, float *dbA,
                         float *dB, float *dbB, void *ws, const MlpWs &L, cudaStream_t s, const SeqPar *sp) {
    float *dU = at<float>(ws, L.dU);
    float *partial = at<float>(ws, L.partial);
    float *Yt = at<float>(ws, L.Yt), *dZt = at<float>(ws, L.dZt), *Xt = at<float>(ws, L.Xt),
          *dUt = at<float>(ws, L.dUt);
    const int64_t Tp = pad4(T);
    const int64_t fw = pre_width(act, f);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f),
              fwi = static_cast<int>(fw);
    const bool glu = act == Act::SwiGLU;
    tpce_status st;
    {
        Operand a{dZ, T, h, h};  // K-major [T, h]
        Operand b{B, f, h, h};   // K-major: N = f rows, K = h columns
        const OutView o[1] = {{dU, T, fw, fw}};
        const OutView in[1] = {{const_cast<float *>(U), T, fw, fw}};  // read by TMA, never written
        const char *nm = glu ? "swiglu_bwd_dY_swiglu_grad" : "mlp_bwd_dY_gelu_grad";
        if (!glu)
            st = sp ? launch_gemm<float, 128, false, false, EpiGeluGrad<float>, kChunkA>(
                          nm, a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {}, s, true, 0, sp->dz)
                    : launch_gemm<float, 128, false, false, EpiGeluGrad<float>>(nm, a, b, o, in, Ti, fi, hi, 0, 0, 0, 0,
                                                                                {}, s);
        else
            st = sp ? launch_gemm<float, 128, false, false, EpiSwiGluGrad<float>, kChunkA>(
                          nm, a, b, o, in, Ti, fi, hi, 0, 0, 0, 0, {fi}, s, true, 0, sp->dz)
                    : launch_gemm<float, 128, false, false, EpiSwiGluGrad<float>>(nm, a, b, o, in, Ti, fi, hi, 0, 0, 0,
                                                                                  0, {fi}, s);
        if (st != TPCE_OK) return st;
    }
    if ((st = transpose_f32(Y, T, f, f, Yt, Tp, s)) != TPCE_OK) return st;
    if (sp) {
        // the gathered dZ^T and X^T, one sequence chunk (a column block) at a time
        for (int c = 0; c < sp->dz->count; ++c) {
            const int64_t r0 = c * sp->dz->rows;
            st = transpose_f32(static_cast<const float *>(sp->dz->ptrs[c]), sp->dz->rows, h, h, dZt + r0, Tp, s);
            if (st != TPCE_OK) return st;
            st = transpose_f32(static_cast<const float *>(sp->x->ptrs[c]), sp->x->rows, h, h, Xt + r0, Tp, s);
            if (st != TPCE_OK) return st;
        }
    } else {
        if ((st = transpose_f32(dZ, T, h, h, dZt, Tp, s)) != TPCE_OK) return st;
        if ((st = transpose_f32(X, T, h, h, Xt, Tp, s)) != TPCE_OK) return st;
    }
    if ((st = transpose_f32(dU, T, fw, fw, dUt, Tp, s)) != TPCE_OK) return st;
    {
        Operand a{Yt, f, T, Tp};   // K-major: M = f rows, K = T columns
        Operand b{dZt, h, T, Tp};  // K-major: N = h rows, K = T columns
        const OutView o[1] = {{dB, f, h, h}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>(glu ? "swiglu_bwd_dW2" : "mlp_bwd_dB", a, b, o,
                                                                    nullptr, fi, hi, Ti, 0, 0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    {
        Operand a{Xt, h, T, Tp};    // K-major: M = h rows, K = T columns
        Operand b{dUt, fw, T, Tp};  // K-major: N = fw rows, K = T columns
        const OutView o[1] = {{dA, h, fw, fw}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>(glu ? "swiglu_bwd_dW1" : "mlp_bwd_dA", a, b, o,
                                                                    nullptr, hi, fwi, Ti, 0, 0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    {
        Operand a{dU, T, fw, fw};  // K-major [T, fw]
        Operand b{A, h, fw, fw};   // K-major: N = h rows, K = fw columns
        const OutView o[1] = {{dX, T, h, h}};
        const char *nm = glu ? "swiglu_bwd_dX_shard_sum" : "mlp_bwd_dX_shard_sum";
        st = sp ? launch_gemm<float, 128, false, false, EpiStore<float>, kChunkC>(
                      nm, a, b, o, nullptr, Ti, hi, fwi, 0, 0, 0, 0, {nullptr}, s, true, 0, sp->out)
                : launch_gemm<float, 128, false, false, EpiStore<float>>(nm, a, b, o, nullptr, Ti, hi, fwi, 0, 0, 0, 0,
                                                                         {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    if (dbA && (st = colsum(1, dU, T, fw, fw, dbA, partial, s)) != TPCE_OK) return st;
    if (dbB) {
        st = sp ? colsum_chunks(1, sp->dz->ptrs, sp->dz->count, sp->dz->rows, h, h, dbB, partial, s)
                : colsum(1, dZ, T, h, h, dbB, partial, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
}

// ---------------------------------------------------------------- entry points
size_t workspace_bytes(Act act, int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (check_mlp_shape(act, T, h, f, t, dtype) != TPCE_OK) return 0;
    return mlp_ws_layout(act, T, h, f, dtype).total;
}

// With sp, X and Z come as sequence chunks (already validated) and X, Z are unused.
tpce_status forward(Act act, const void *X, const void *A, const float *bA, const void *B, const float *bB, int64_t T,
                    int64_t h, int64_t f, int t, int dtype, void *Z, void *U, void *Y, void *ws, size_t ws_bytes,
                    void *stream, const SeqPar *sp = nullptr) {
    tpce_status st = check_mlp_shape(act, T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;  // no tokens: nothing to compute (token tensors may be NULL)
    if (!A || !B || !U || !Y || (!sp && (!X || !Z))) return TPCE_ERR_INVALID;
    for (const void *p : {X, A, B, static_cast<const void *>(Z), static_cast<const void *>(U),
                          static_cast<const void *>(Y), static_cast<const void *>(bA), static_cast<const void *>(bB),
                          static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TPCE_BF16) {
        const TailScratch tail = tail_of(ws, ws_bytes);  // optional: splits the last wave's tiles
        return forward_bf16(act, X, A, bA, B, bB, T, h, f, Z, U, Y, s, sp, &tail);
    }
    const MlpWs L = mlp_ws_layout(act, T, h, f, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    return forward_f32(act, static_cast<const float *>(X), static_cast<const float *>(A), bA,
                       static_cast<const float *>(B), bB, T, h, f, static_cast<float *>(Z), static_cast<float *>(U),
                       static_cast<float *>(Y), ws, L, s, sp);
}

// With sp, dZ, X and dX come as sequence chunks (already validated) and are unused.
tpce_status backward(Act act, const void *dZ, const void *X, const void *A, const void *B, const void *U,
                     const void *Y, int64_t T, int64_t h, int64_t f, int t, int dtype, void *dX, void *dA, float *dbA,
                     void *dB, float *dbB, void *ws, size_t ws_bytes, void *stream, const SeqPar *sp = nullptr) {
    tpce_status st = check_mlp_shape(act, T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (!A || !B || !dA || !dB) return TPCE_ERR_INVALID;
    if (T > 0 && (!U || !Y || (!sp && (!dZ || !X || !dX)))) return TPCE_ERR_INVALID;
    for (const void *p : {dZ, X, A, B, U, Y, static_cast<const void *>(dX), static_cast<const void *>(dA),
                          static_cast<const void *>(dB), static_cast<const void *>(dbA),
                          static_cast<const void *>(dbB), static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t esz = dtype == TPCE_F32 ? 4 : 2;
    const int64_t fw = pre_width(act, f);
    if (T == 0) {
        // no tokens: every weight and bias gradient is an empty sum
        if (cudaMemsetAsync(dA, 0, static_cast<size_t>(h) * fw * esz, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (cudaMemsetAsync(dB, 0, static_cast<size_t>(f) * h * esz, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbA && cudaMemsetAsync(dbA, 0, sizeof(float) * fw, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbB && cudaMemsetAsync(dbB, 0, sizeof(float) * h, s) != cudaSuccess) return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const MlpWs L = mlp_ws_layout(act, T, h, f, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    if (dtype == TPCE_BF16)
        return backward_bf16(act, dZ, X, A, B, U, Y, T, h, f, dX, dA, dbA, dB, dbB, ws, L, s, sp);
    return backward_f32(act, static_cast<const float *>(dZ), static_cast<const float *>(X),
                        static_cast<const float *>(A), static_cast<const float *>(B), static_cast<const float *>(U),
                        static_cast<const float *>(Y), T, h, f, static_cast<float *>(dX), static_cast<float *>(dA), dbA,
                        static_cast<float *>(dB), dbB, ws, L, s, sp);
}

// Sequence chunks of a [T, h] activation: t buffers of T/t rows, each row a
// whole number of 128-row boxes so that no tile row-block straddles two.
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

tpce_status forward_sp(Act act, const void *const *X_chunks, const void *A, const float *bA, const void *B,
                       const float *bB, int64_t T, int64_t h, int64_t f, int t, int dtype, void *const *Z_chunks,
                       void *U, void *Y, void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_mlp_shape(act, T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;
    Chunks xc{}, zc{};
    if ((st = check_chunks(X_chunks, T, t, xc)) != TPCE_OK) return st;
    if ((st = check_chunks(reinterpret_cast<const void *const *>(Z_chunks), T, t, zc)) != TPCE_OK) return st;
    const SeqPar sp{&xc, nullptr, &zc};
    return forward(act, nullptr, A, bA, B, bB, T, h, f, t, dtype, nullptr, U, Y, ws, ws_bytes, stream, &sp);
}

tpce_status backward_sp(Act act, const void *const *dZ_chunks, const void *const *X_chunks, const void *A,
                        const void *B, const void *U, const void *Y, int64_t T, int64_t h, int64_t f, int t, int dtype,
                        void *const *dX_chunks, void *dA, float *dbA, void *dB, float *dbB, void *ws, size_t ws_bytes,
                        void *stream) {
    tpce_status st = check_mlp_shape(act, T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0)  // no tokens: the dense path zeroes the weight and bias gradients
        return backward(act, nullptr, nullptr, A, B, nullptr, nullptr, 0, h, f, t, dtype, nullptr, dA, dbA, dB, dbB,
                        ws, ws_bytes, stream);
    Chunks dzc{}, xc{}, dxc{};
    if ((st = check_chunks(dZ_chunks, T, t, dzc)) != TPCE_OK) return st;
    if ((st = check_chunks(X_chunks, T, t, xc)) != TPCE_OK) return st;
    if ((st = check_chunks(reinterpret_cast<const void *const *>(dX_chunks), T, t, dxc)) != TPCE_OK) return st;
    const SeqPar sp{&xc, &dzc, &dxc};
    return backward(act, nullptr, nullptr, A, B, U, Y, T, h, f, t, dtype, nullptr, dA, dbA, dB, dbB, ws, ws_bytes,
                    stream, &sp);
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_mlp_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    return workspace_bytes(Act::GeLU, T, h, f, t, dtype);
}

extern "C" tpce_status tp_mlp_forward(const void *X, const void *A, const float *bA, const void *B, const float *bB,
                                      int64_t T, int64_t h, int64_t f, int t, int dtype, void *Z, void *U, void *Y,
                                      void *ws, size_t ws_bytes, void *stream) {
    return forward(Act::GeLU, X, A, bA, B, bB, T, h, f, t, dtype, Z, U, Y, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_mlp_backward(const void *dZ, const void *X, const void *A, const void *B, const void *U,
                                       const void *Y, int64_t T, int64_t h, int64_t f, int t, int dtype, void *dX,
                                       void *dA, float *dbA, void *dB, float *dbB, void *ws, size_t ws_bytes,
                                       void *stream) {
    return backward(Act::GeLU, dZ, X, A, B, U, Y, T, h, f, t, dtype, dX, dA, dbA, dB, dbB, ws, ws_bytes, stream);
}

extern "C" size_t tpce_swiglu_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    return workspace_bytes(Act::SwiGLU, T, h, f, t, dtype);
}

extern "C" tpce_status tp_swiglu_forward(const void *X, const void *W1, const float *b1, const void *W2,
                                         const float *b2, int64_t T, int64_t h, int64_t f, int t, int dtype, void *Z,
                                         void *GU, void *Y, void *ws, size_t ws_bytes, void *stream) {
    return forward(Act::SwiGLU, X, W1, b1, W2, b2, T, h, f, t, dtype, Z, GU, Y, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_swiglu_backward(const void *dZ, const void *X, const void *W1, const void *W2,
                                          const void *GU, const void *Y, int64_t T, int64_t h, int64_t f, int t,
                                          int dtype, void *dX, void *dW1, float *db1, void *dW2, float *db2, void *ws,
                                          size_t ws_bytes, void *stream) {
    return backward(Act::SwiGLU, dZ, X, W1, W2, GU, Y, T, h, f, t, dtype, dX, dW1, db1, dW2, db2, ws, ws_bytes,
                    stream);
}

extern "C" tpce_status tp_mlp_forward_sp(const void *const *X_chunks, const void *A, const float *bA, const void *B,
                                         const float *bB, int64_t T, int64_t h, int64_t f, int t, int dtype,
                                         void *const *Z_chunks, void *U, void *Y, void *ws, size_t ws_bytes,
                                         void *stream) {
    return forward_sp(Act::GeLU, X_chunks, A, bA, B, bB, T, h, f, t, dtype, Z_chunks, U, Y, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_mlp_backward_sp(const void *const *dZ_chunks, const void *const *X_chunks, const void *A,
                                          const void *B, const void *U, const void *Y, int64_t T, int64_t h, int64_t f,
                                          int t, int dtype, void *const *dX_chunks, void *dA, float *dbA, void *dB,
                                          float *dbB, void *ws, size_t ws_bytes, void *stream) {
    return backward_sp(Act::GeLU, dZ_chunks, X_chunks, A, B, U, Y, T, h, f, t, dtype, dX_chunks, dA, dbA, dB, dbB, ws,
                       ws_bytes, stream);
}

extern "C" tpce_status tp_swiglu_forward_sp(const void *const *X_chunks, const void *W1, const float *b1,
                                            const void *W2, const float *b2, int64_t T, int64_t h, int64_t f, int t,
                                            int dtype, void *const *Z_chunks, void *GU, void *Y, void *ws,
                                            size_t ws_bytes, void *stream) {
    return forward_sp(Act::SwiGLU, X_chunks, W1, b1, W2, b2, T, h, f, t, dtype, Z_chunks, GU, Y, ws, ws_bytes, stream);
}

extern "C" tpce_status tp_swiglu_backward_sp(const void *const *dZ_chunks, const void *const *X_chunks,
                                             const void *W1, const void *W2, const void *GU, const void *Y, int64_t T,
                                             int64_t h, int64_t f, int t, int dtype, void *const *dX_chunks,
                                             void *dW1, float *db1, void *dW2, float *db2, void *ws, size_t ws_bytes,
                                             void *stream) {
    return backward_sp(Act::SwiGLU, dZ_chunks, X_chunks, W1, W2, GU, Y, T, h, f, t, dtype, dX_chunks, dW1, db1, dW2,
                       db2, ws, ws_bytes, stream);
}
