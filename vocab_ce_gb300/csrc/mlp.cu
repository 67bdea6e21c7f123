// mlp.cu -- tp_mlp_forward / tp_mlp_backward: the Megatron 1D tensor-parallel
// MLP block with its t shards laid out on one GPU.
//
// Forward ("Mathematical Foundations of Megatron-LM 1D Slicing", sections
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
// bf16 tensors use the bf16 tensor-core path with operands read in place in
// either major order. fp32 tensors use the tf32 path, whose operands are
// K-major: the operands stored the other way (A and B in the forward, Y, dZ,
// X, dU in the weight gradients) are first transposed into the workspace.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

constexpr int64_t kMaxDim = INT_MAX - 1024;  // kernel coordinates are 32-bit

tpce_status check_mlp_shape(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (dtype != TPCE_BF16 && dtype != TPCE_F32) return TPCE_ERR_INVALID;
    if (T < 0 || h < 8 || f < 1 || t < 1) return TPCE_ERR_SHAPE;
    if (T > kMaxDim || h > kMaxDim || f > kMaxDim) return TPCE_ERR_SHAPE;
    if (h % 8 != 0) return TPCE_ERR_SHAPE;           // 16-byte row pitch
    if (f % t != 0) return TPCE_ERR_SHAPE;           // equal shards
    if ((f / t) % 64 != 0) return TPCE_ERR_SHAPE;    // a shard is whole 64-wide blocks
    if (dtype == TPCE_F32 && (T + 31) / 32 > 65535) return TPCE_ERR_SHAPE;  // transpose grid
    return TPCE_OK;
}

inline int64_t pad4(int64_t x) { return (x + 3) / 4 * 4; }  // fp32 rows padded to 16 bytes

// Workspace layout. bf16: dU [T, f] and the column-sum partials. fp32 adds the
// transposed operands of the tf32 path: A^T, B^T (forward), Y^T, dZ^T, X^T,
// dU^T (backward), the token-major ones with rows padded to a multiple of 4.
struct MlpWs {
    size_t dU, partial, At, Bt, Yt, dZt, Xt, dUt, total;
};

MlpWs mlp_ws_layout(int64_t T, int64_t h, int64_t f, int dtype) {
    MlpWs L{};
    const size_t esz = dtype == TPCE_F32 ? 4 : 2;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = round_up(off + bytes, 256);
        return at;
    };
    L.dU = take(static_cast<size_t>(T) * f * esz);
    const size_t pf = std::max(colsum_partial_floats(T, f), colsum_partial_floats(T, h));
    L.partial = take(pf * sizeof(float));
    if (dtype == TPCE_F32) {
        const size_t Tp = static_cast<size_t>(pad4(T));
        L.At = take(static_cast<size_t>(f) * h * 4);
        L.Bt = take(static_cast<size_t>(h) * f * 4);
        L.Yt = take(static_cast<size_t>(f) * Tp * 4);
        L.dZt = take(static_cast<size_t>(h) * Tp * 4);
        L.Xt = take(static_cast<size_t>(h) * Tp * 4);
        L.dUt = take(static_cast<size_t>(f) * Tp * 4);
    }
    L.total = off;
    return L;
}

template <typename T>
T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(static_cast<uint8_t *>(ws) + off);
}

// ---------------------------------------------------------------- bf16 path
tpce_status forward_bf16(const void *X, const void *A, const float *bA, const void *B, const float *bB, int64_t T,
                         int64_t h, int64_t f, void *Z, void *U, void *Y, cudaStream_t s) {
    using bf = __nv_bfloat16;
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    // GEMM1 (column-parallel): U = X A + bA, Y = GeLU(U)
    Operand a{X, T, h, h};  // K-major [T, h]
    Operand b{A, h, f, f};  // MN-major: K = h rows, N = f columns
    const OutView o1[2] = {{U, T, f, f}, {Y, T, f, f}};
    tpce_status st = launch_gemm_auto<bf, false, true, EpiBiasGelu<bf>, kBN192 | kBN256>(
        "mlp_fwd_gemm1_bias_gelu", a, b, o1, nullptr, Ti, fi, hi, 0, 0, 0, 0, {bA}, s);
    if (st != TPCE_OK) return st;
    // GEMM2 (row-parallel) + g: Z = sum_i Y_i B_i + bB
    Operand a2{Y, T, f, f};  // K-major [T, f]
    Operand b2{B, f, h, h};  // MN-major: K = f rows, N = h columns
    const OutView o2[1] = {{Z, T, h, h}};
    return launch_gemm_auto<bf, false, true, EpiStore<bf>, kBN192 | kBN256>("mlp_fwd_gemm2_shard_sum", a2, b2, o2, nullptr,
                                                                             Ti, hi, fi, 0, 0, 0, 0, {bB}, s);
}

tpce_status backward_bf16(const void *dZ, const void *X, const void *A, const void *B, const void *U,
                          const void *Y, int64_t T, int64_t h, int64_t f, void *dX, void *dA, float *dbA, void *dB,
                          float *dbB, void *ws, const MlpWs &L, cudaStream_t s) {
    using bf = __nv_bfloat16;
    bf *dU = at<bf>(ws, L.dU);
    float *partial = at<float>(ws, L.partial);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    tpce_status st;
    // g* is the identity: every shard reads the same dZ.
    // dY_i = dZ B_i^T, fused with dU_i = dY_i (.) GeLU'(U_i)
    {
        Operand a{dZ, T, h, h};  // K-major [T, h]
        Operand b{B, f, h, h};   // K-major: N = f rows, K = h columns
        const OutView o[1] = {{dU, T, f, f}};
        const OutView in[1] = {{const_cast<void *>(U), T, f, f}};  // read by TMA, never written
        st = launch_gemm_auto<bf, false, false, EpiGeluGrad<bf>, kBN192 | kBN256>("mlp_bwd_dY_gelu_grad", a, b, o, in,
                                                                                   Ti, fi, hi, 0, 0, 0, 0, {}, s);
        if (st != TPCE_OK) return st;
    }
    // dB_i = Y_i^T dZ
    {
        Operand a{Y, T, f, f};   // MN-major: K = T rows, M = f columns
        Operand b{dZ, T, h, h};  // MN-major: K = T rows, N = h columns
        const OutView o[1] = {{dB, f, h, h}};
        st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>("mlp_bwd_dB", a, b, o, nullptr, fi, hi, Ti, 0,
                                                                              0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    // dA_i = X^T dU_i
    {
        Operand a{X, T, h, h};   // MN-major: K = T rows, M = h columns
        Operand b{dU, T, f, f};  // MN-major: K = T rows, N = f columns
        const OutView o[1] = {{dA, h, f, f}};
        st = launch_gemm_auto<bf, true, true, EpiStore<bf>, kBN192 | kBN256>("mlp_bwd_dA", a, b, o, nullptr, hi, fi, Ti, 0,
                                                                              0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    // f*: dX = sum_i dU_i A_i^T, the shard sum taken in the accumulator
    {
        Operand a{dU, T, f, f};  // K-major [T, f]
        Operand b{A, h, f, f};   // K-major: N = h rows, K = f columns
        const OutView o[1] = {{dX, T, h, h}};
        st = launch_gemm_auto<bf, false, false, EpiStore<bf>, kBN192 | kBN256>("mlp_bwd_dX_shard_sum", a, b, o, nullptr, Ti,
                                                                                hi, fi, 0, 0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    if (dbA && (st = colsum(0, dU, T, f, f, dbA, partial, s)) != TPCE_OK) return st;
    if (dbB && (st = colsum(0, dZ, T, h, h, dbB, partial, s)) != TPCE_OK) return st;
    return TPCE_OK;
}

// ---------------------------------------------------------------- fp32 (tf32) path
tpce_status forward_f32(const float *X, const float *A, const float *bA, const float *B, const float *bB, int64_t T,
                        int64_t h, int64_t f, float *Z, float *U, float *Y, void *ws, const MlpWs &L,
                        cudaStream_t s) {
    float *At = at<float>(ws, L.At), *Bt = at<float>(ws, L.Bt);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    tpce_status st = transpose_f32(A, h, f, f, At, h, s);  // A^T [f, h]
    if (st != TPCE_OK) return st;
    if ((st = transpose_f32(B, f, h, h, Bt, f, s)) != TPCE_OK) return st;  // B^T [h, f]
    {
        Operand a{X, T, h, h};    // K-major [T, h]
        Operand b{At, f, h, h};   // K-major: N = f rows, K = h columns
        const OutView o[2] = {{U, T, f, f}, {Y, T, f, f}};
        st = launch_gemm<float, 128, false, false, EpiBiasGelu<float>>("mlp_fwd_gemm1_bias_gelu", a, b, o, nullptr, Ti, fi,
                                                                       hi, 0, 0, 0, 0, {bA}, s);
        if (st != TPCE_OK) return st;
    }
    Operand a2{Y, T, f, f};   // K-major [T, f]
    Operand b2{Bt, h, f, f};  // K-major: N = h rows, K = f columns
    const OutView o2[1] = {{Z, T, h, h}};
    return launch_gemm<float, 128, false, false, EpiStore<float>>("mlp_fwd_gemm2_shard_sum", a2, b2, o2, nullptr, Ti, hi, fi,
                                                                  0, 0, 0, 0, {bB}, s);
}

tpce_status backward_f32(const float *dZ, const float *X, const float *A, const float *B, const float *U,
                         const float *Y, int64_t T, int64_t h, int64_t f, float *dX, float *dA, float *dbA,
                         float *dB, float *dbB, void *ws, const MlpWs &L, cudaStream_t s) {
    float *dU = at<float>(ws, L.dU);
    float *partial = at<float>(ws, L.partial);
    float *Yt = at<float>(ws, L.Yt), *dZt = at<float>(ws, L.dZt), *Xt = at<float>(ws, L.Xt),
          *dUt = at<float>(ws, L.dUt);
    const int64_t Tp = pad4(T);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);
    tpce_status st;
    {
        Operand a{dZ, T, h, h};  // K-major [T, h]
        Operand b{B, f, h, h};   // K-major: N = f rows, K = h columns
        const OutView o[1] = {{dU, T, f, f}};
        const OutView in[1] = {{const_cast<float *>(U), T, f, f}};  // read by TMA, never written
        st = launch_gemm<float, 128, false, false, EpiGeluGrad<float>>("mlp_bwd_dY_gelu_grad", a, b, o, in, Ti, fi,
                                                                       hi, 0, 0, 0, 0, {}, s);
        if (st != TPCE_OK) return st;
    }
    if ((st = transpose_f32(Y, T, f, f, Yt, Tp, s)) != TPCE_OK) return st;
    if ((st = transpose_f32(dZ, T, h, h, dZt, Tp, s)) != TPCE_OK) return st;
    if ((st = transpose_f32(X, T, h, h, Xt, Tp, s)) != TPCE_OK) return st;
    if ((st = transpose_f32(dU, T, f, f, dUt, Tp, s)) != TPCE_OK) return st;
    {
        Operand a{Yt, f, T, Tp};   // K-major: M = f rows, K = T columns
        Operand b{dZt, h, T, Tp};  // K-major: N = h rows, K = T columns
        const OutView o[1] = {{dB, f, h, h}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>("mlp_bwd_dB", a, b, o, nullptr, fi, hi, Ti, 0, 0, 0, 0,
                                                                    {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    {
        Operand a{Xt, h, T, Tp};   // K-major: M = h rows, K = T columns
        Operand b{dUt, f, T, Tp};  // K-major: N = f rows, K = T columns
        const OutView o[1] = {{dA, h, f, f}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>("mlp_bwd_dA", a, b, o, nullptr, hi, fi, Ti, 0, 0, 0, 0,
                                                                    {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    {
        Operand a{dU, T, f, f};  // K-major [T, f]
        Operand b{A, h, f, f};   // K-major: N = h rows, K = f columns
        const OutView o[1] = {{dX, T, h, h}};
        st = launch_gemm<float, 128, false, false, EpiStore<float>>("mlp_bwd_dX_shard_sum", a, b, o, nullptr, Ti, hi, fi, 0,
                                                                    0, 0, 0, {nullptr}, s);
        if (st != TPCE_OK) return st;
    }
    if (dbA && (st = colsum(1, dU, T, f, f, dbA, partial, s)) != TPCE_OK) return st;
    if (dbB && (st = colsum(1, dZ, T, h, h, dbB, partial, s)) != TPCE_OK) return st;
    return TPCE_OK;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_mlp_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (check_mlp_shape(T, h, f, t, dtype) != TPCE_OK) return 0;
    return mlp_ws_layout(T, h, f, dtype).total;
}

extern "C" tpce_status tp_mlp_forward(const void *X, const void *A, const float *bA, const void *B, const float *bB,
                                      int64_t T, int64_t h, int64_t f, int t, int dtype, void *Z, void *U, void *Y,
                                      void *ws, size_t ws_bytes, void *stream) {
    tpce_status st = check_mlp_shape(T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;  // no tokens: nothing to compute (token tensors may be NULL)
    if (!X || !A || !B || !Z || !U || !Y) return TPCE_ERR_INVALID;
    for (const void *p : {X, A, B, static_cast<const void *>(Z), static_cast<const void *>(U),
                          static_cast<const void *>(Y), static_cast<const void *>(bA), static_cast<const void *>(bB),
                          static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == TPCE_BF16) return forward_bf16(X, A, bA, B, bB, T, h, f, Z, U, Y, s);
    const MlpWs L = mlp_ws_layout(T, h, f, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    return forward_f32(static_cast<const float *>(X), static_cast<const float *>(A), bA,
                       static_cast<const float *>(B), bB, T, h, f, static_cast<float *>(Z), static_cast<float *>(U),
                       static_cast<float *>(Y), ws, L, s);
}

extern "C" tpce_status tp_mlp_backward(const void *dZ, const void *X, const void *A, const void *B, const void *U,
                                       const void *Y, int64_t T, int64_t h, int64_t f, int t, int dtype, void *dX,
                                       void *dA, float *dbA, void *dB, float *dbB, void *ws, size_t ws_bytes,
                                       void *stream) {
    tpce_status st = check_mlp_shape(T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (!A || !B || !dA || !dB) return TPCE_ERR_INVALID;
    if (T > 0 && (!dZ || !X || !U || !Y || !dX)) return TPCE_ERR_INVALID;
    for (const void *p : {dZ, X, A, B, U, Y, static_cast<const void *>(dX), static_cast<const void *>(dA),
                          static_cast<const void *>(dB), static_cast<const void *>(dbA),
                          static_cast<const void *>(dbB), static_cast<const void *>(ws)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t esz = dtype == TPCE_F32 ? 4 : 2;
    if (T == 0) {
        // no tokens: every weight and bias gradient is an empty sum
        if (cudaMemsetAsync(dA, 0, static_cast<size_t>(h) * f * esz, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (cudaMemsetAsync(dB, 0, static_cast<size_t>(f) * h * esz, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbA && cudaMemsetAsync(dbA, 0, sizeof(float) * f, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbB && cudaMemsetAsync(dbB, 0, sizeof(float) * h, s) != cudaSuccess) return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const MlpWs L = mlp_ws_layout(T, h, f, dtype);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    if (dtype == TPCE_BF16) return backward_bf16(dZ, X, A, B, U, Y, T, h, f, dX, dA, dbA, dB, dbB, ws, L, s);
    return backward_f32(static_cast<const float *>(dZ), static_cast<const float *>(X), static_cast<const float *>(A),
                        static_cast<const float *>(B), static_cast<const float *>(U), static_cast<const float *>(Y),
                        T, h, f, static_cast<float *>(dX), static_cast<float *>(dA), dbA, static_cast<float *>(dB),
                        dbB, ws, L, s);
}
