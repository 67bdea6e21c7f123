// gemm_launch.cuh -- host-side launch of tc_gemm_kernel: tensor maps, tile
// grid, rasterisation and the persistent grid size.
#pragma once

#include <algorithm>
#include <mutex>

#include "gemm.cuh"
#include "host.h"

namespace tpce {
// Internal linkage: every translation unit gets its own kernels and launch
// state (a kernel instantiated in two units is two device functions).
namespace {

// An operand as it sits in memory (row-major, row pitch `ld` elements).
// K-major operand: `rows` = extent of the output dimension it feeds (M for A,
// N for B), `cols` = contraction extent. MN-major operand: `rows` =
// contraction extent, `cols` = output-dimension extent.
struct Operand {
    const void *ptr;
    int64_t rows, cols, ld;
};

// Tiles are walked in groups of `group_m` row-blocks, row-block fastest, so
// the CTAs of one wave share a few A and B panels in L2.
inline int pick_group_m(int tiles_m) { return std::max(1, std::min(tiles_m, 16)); }

// Raise the kernel's dynamic shared-memory limit, once per device. `done` must
// be distinct per kernel instantiation (kernels of equal signature share a
// function type), so each caller passes its own flags.
template <class K>
inline tpce_status set_smem_attr(K kern, uint32_t bytes, bool (&done)[64], std::mutex &mu) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fail(TPCE_ERR_CUDA, "cudaGetDevice");
    std::lock_guard<std::mutex> g(mu);
    if (!done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
        if (e != cudaSuccess) return fail_cuda(e, "cudaFuncSetAttribute");
        done[dev] = true;
    }
    return TPCE_OK;
}

// D = A * B with the epilogue Epi. Offsets shift the operands' coordinates
// inside their tensor maps (used to address one vocabulary chunk of E).
template <int BN, bool A_MN, bool B_MN, class Epi>
tpce_status launch_gemm(const char *name, const Operand &a, const Operand &b, int M, int N, int K, int a_off_mn,
                        int a_off_k, int b_off_mn, int b_off_k, const typename Epi::Params &ep,
                        cudaStream_t stream, bool timed = true) {
    using Cfg = TileCfg<BN>;
    if (M <= 0 || N <= 0 || K <= 0) return TPCE_ERR_SHAPE;
    CUtensorMap ta, tb;
    bool ok = A_MN ? make_tmap_bf16(&ta, a.ptr, a.cols, a.rows, a.ld, 64, 64)
                   : make_tmap_bf16(&ta, a.ptr, a.cols, a.rows, a.ld, 64, kBM);
    ok = ok && (B_MN ? make_tmap_bf16(&tb, b.ptr, b.cols, b.rows, b.ld, 64, 64)
                     : make_tmap_bf16(&tb, b.ptr, b.cols, b.rows, b.ld, 64, BN));
    if (!ok) return fail(TPCE_ERR_CUDA, "cuTensorMapEncodeTiled rejected an operand of %s", name);

    GemmShape s;
    s.M = M;
    s.N = N;
    s.K = K;
    s.tiles_m = (M + kBM - 1) / kBM;
    s.tiles_n = (N + BN - 1) / BN;
    s.k_blocks = (K + kBK - 1) / kBK;
    s.group_m = pick_group_m(s.tiles_m);
    s.a_off_mn = a_off_mn;
    s.a_off_k = a_off_k;
    s.b_off_mn = b_off_mn;
    s.b_off_k = b_off_k;

    auto kern = tc_gemm_kernel<BN, A_MN, B_MN, Epi>;
    static std::mutex attr_mu;
    static bool attr_done[64] = {};
    tpce_status st = set_smem_attr(kern, Cfg::kSmemBytes, attr_done, attr_mu);
    if (st != TPCE_OK) return st;
    const int sms = num_sms();
    uint32_t *err = device_error_word();
    if (sms <= 0 || err == nullptr) return fail(TPCE_ERR_CUDA, "device query failed (%s)", name);
    const int64_t tiles = static_cast<int64_t>(s.tiles_m) * s.tiles_n;
    const int grid = static_cast<int>(std::min<int64_t>(tiles, sms));
    KernelTimer timer(timed ? name : nullptr, stream);
    kern<<<grid, kThreads, Cfg::kSmemBytes, stream>>>(ta, tb, s, ep, err);
    return check_launch(name);
}

}  // namespace
}  // namespace tpce
