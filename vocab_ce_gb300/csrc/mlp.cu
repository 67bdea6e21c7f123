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
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <climits>

#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {
namespace {

constexpr int64_t kMaxDim = INT_MAX - 1024;  // kernel coordinates are 32-bit

tpce_status check_mlp_shape(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (dtype == TPCE_F32) return TPCE_ERR_UNSUPPORTED;
    if (dtype != TPCE_BF16) return TPCE_ERR_INVALID;
    if (T < 0 || h < 8 || f < 1 || t < 1) return TPCE_ERR_SHAPE;
    if (T > kMaxDim || h > kMaxDim || f > kMaxDim) return TPCE_ERR_SHAPE;
    if (h % 8 != 0) return TPCE_ERR_SHAPE;           // 16-byte row pitch
    if (f % t != 0) return TPCE_ERR_SHAPE;           // equal shards
    if ((f / t) % 64 != 0) return TPCE_ERR_SHAPE;    // a shard is whole 64-wide blocks
    return TPCE_OK;
}

struct MlpWs {
    size_t dU, partial, total;
};

MlpWs mlp_ws_layout(int64_t T, int64_t h, int64_t f) {
    MlpWs L;
    L.dU = 0;
    L.partial = round_up(static_cast<size_t>(T) * f * 2, 256);
    const size_t pf = std::max(colsum_partial_floats(T, f), colsum_partial_floats(T, h));
    L.total = L.partial + round_up(pf * sizeof(float), 256);
    return L;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" size_t tpce_mlp_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype) {
    if (check_mlp_shape(T, h, f, t, dtype) != TPCE_OK) return 0;
    return mlp_ws_layout(T, h, f).total;
}

extern "C" tpce_status tp_mlp_forward(const void *X, const void *A, const float *bA, const void *B, const float *bB,
                                      int64_t T, int64_t h, int64_t f, int t, int dtype, void *Z, void *U, void *Y,
                                      void *ws, size_t ws_bytes, void *stream) {
    (void)ws;
    (void)ws_bytes;
    tpce_status st = check_mlp_shape(T, h, f, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;  // no tokens: nothing to compute (token tensors may be NULL)
    if (!X || !A || !B || !Z || !U || !Y) return TPCE_ERR_INVALID;
    for (const void *p : {X, A, B, static_cast<const void *>(Z), static_cast<const void *>(U),
                          static_cast<const void *>(Y), static_cast<const void *>(bA), static_cast<const void *>(bB)})
        if (!aligned16(p)) return TPCE_ERR_ALIGN;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);

    // GEMM1 (column-parallel): U = X A + bA, Y = GeLU(U)
    {
        Operand a{X, T, h, h};  // K-major [T, h]
        Operand b{A, h, f, f};  // MN-major: K = h rows, N = f columns
        EpiBiasGelu::Params ep{static_cast<__nv_bfloat16 *>(U), static_cast<__nv_bfloat16 *>(Y), bA, f};
        st = launch_gemm<256, false, true, EpiBiasGelu>("mlp_fwd_gemm1_bias_gelu", a, b, Ti, fi, hi, 0, 0, 0, 0,
                                                         ep, s);
        if (st != TPCE_OK) return st;
    }
    // GEMM2 (row-parallel) + g: Z = sum_i Y_i B_i + bB
    {
        Operand a{Y, T, f, f};  // K-major [T, f]
        Operand b{B, f, h, h};  // MN-major: K = f rows, N = h columns
        EpiStore::Params ep{static_cast<__nv_bfloat16 *>(Z), bB, h};
        st = launch_gemm<256, false, true, EpiStore>("mlp_fwd_gemm2_shard_sum", a, b, Ti, hi, fi, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
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
    if (T == 0) {
        // no tokens: every weight and bias gradient is an empty sum
        if (cudaMemsetAsync(dA, 0, static_cast<size_t>(h) * f * 2, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (cudaMemsetAsync(dB, 0, static_cast<size_t>(f) * h * 2, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbA && cudaMemsetAsync(dbA, 0, sizeof(float) * f, s) != cudaSuccess) return TPCE_ERR_CUDA;
        if (dbB && cudaMemsetAsync(dbB, 0, sizeof(float) * h, s) != cudaSuccess) return TPCE_ERR_CUDA;
        return TPCE_OK;
    }
    const MlpWs L = mlp_ws_layout(T, h, f);
    if (!ws || ws_bytes < L.total) return TPCE_ERR_WORKSPACE;
    __nv_bfloat16 *dU = reinterpret_cast<__nv_bfloat16 *>(static_cast<uint8_t *>(ws) + L.dU);
    float *partial = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + L.partial);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), fi = static_cast<int>(f);

    // g* is the identity: every shard reads the same dZ.
    // dY_i = dZ B_i^T, fused with dU_i = dY_i (.) GeLU'(U_i)
    {
        Operand a{dZ, T, h, h};  // K-major [T, h]
        Operand b{B, f, h, h};   // K-major: N = f rows, K = h columns
        EpiGeluGrad::Params ep{dU, static_cast<const __nv_bfloat16 *>(U), f};
        st = launch_gemm<256, false, false, EpiGeluGrad>("mlp_bwd_dY_gelu_grad", a, b, Ti, fi, hi, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    // dB_i = Y_i^T dZ
    {
        Operand a{Y, T, f, f};   // MN-major: K = T rows, M = f columns
        Operand b{dZ, T, h, h};  // MN-major: K = T rows, N = h columns
        EpiStore::Params ep{static_cast<__nv_bfloat16 *>(dB), nullptr, h};
        st = launch_gemm<256, true, true, EpiStore>("mlp_bwd_dB", a, b, fi, hi, Ti, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    // dA_i = X^T dU_i
    {
        Operand a{X, T, h, h};   // MN-major: K = T rows, M = h columns
        Operand b{dU, T, f, f};  // MN-major: K = T rows, N = f columns
        EpiStore::Params ep{static_cast<__nv_bfloat16 *>(dA), nullptr, f};
        st = launch_gemm<256, true, true, EpiStore>("mlp_bwd_dA", a, b, hi, fi, Ti, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    // f*: dX = sum_i dU_i A_i^T, the shard sum taken in the accumulator
    {
        Operand a{dU, T, f, f};  // K-major [T, f]
        Operand b{A, h, f, f};   // K-major: N = h rows, K = f columns
        EpiStore::Params ep{static_cast<__nv_bfloat16 *>(dX), nullptr, h};
        st = launch_gemm<256, false, false, EpiStore>("mlp_bwd_dX_shard_sum", a, b, Ti, hi, fi, 0, 0, 0, 0, ep, s);
        if (st != TPCE_OK) return st;
    }
    if (dbA) {
        st = colsum_bf16(dU, T, f, f, dbA, partial, s);
        if (st != TPCE_OK) return st;
    }
    if (dbB) {
        st = colsum_bf16(dZ, T, h, h, dbB, partial, s);
        if (st != TPCE_OK) return st;
    }
    return TPCE_OK;
}
