// gemm.cuh -- the tensor-core GEMM behind every contraction of the block.
//
// D[M, N] = sum_k A[m, k] B[k, n] with bf16 operands and an fp32 accumulator
// in tensor memory, followed by a fused epilogue. One persistent CTA per SM
// walks the output tiles; inside a CTA the work is split by warp:
//
//   warp 0      TMA producer: streams 128x64 A and BNx64 B tiles into a ring
//               of shared-memory stages (128-byte swizzle).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN, K=16)
//               into one of two TMEM accumulators; it also owns the TMEM
//               allocation.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one row per thread),
//               apply the fused epilogue, store to global memory, and hand the
//               accumulator back, so the next tile's MMAs overlap this tile's
//               epilogue.
//
// Operands can be K-major (rows of the contraction dimension contiguous) or
// MN-major (the output dimension contiguous): the transposed operands of the
// backward GEMMs (Y^T dZ, X^T dU, dl^T H) are read in place, no transpose pass.
//
// The tile grid's N coordinate of the column-parallel GEMMs is the
// concatenation of the t shards' column ranges, and the K loop of the
// row-parallel GEMMs is the concatenation of the t shards' reduction ranges:
// the accumulator therefore sums the shard partials Z_i (the g operator of
// the Megatron pages) on chip, in fp32.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "ptx.cuh"

namespace tpce {
// Internal linkage: every translation unit gets its own kernels and launch
// state (a kernel instantiated in two units is two device functions).
namespace {

constexpr int kBM = 128;           // tile rows (TMEM lanes)
constexpr int kBK = 64;            // bf16 elements per 128-byte swizzle row
constexpr int kUmmaK = 16;         // K of one tcgen05.mma kind::f16
constexpr int kThreads = 192;      // 6 warps
constexpr uint32_t kMnBlockBytes = 64 * kBK * 2;   // one 64-wide MN block of an MN-major tile

template <int BN>
struct TileCfg {
    static constexpr int kStages = BN == 256 ? 4 : 6;
    static constexpr uint32_t kABytes = kBM * kBK * 2;
    static constexpr uint32_t kBBytes = BN * kBK * 2;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = 2 * BN;           // two accumulators
    static constexpr uint32_t kBarrierBytes = 256;
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + 1024 + kBarrierBytes;
};

// Problem description shared by every role of the kernel.
struct GemmShape {
    int M, N, K;               // output rows, output columns, contraction length
    int tiles_m, tiles_n;      // ceil(M / 128), ceil(N / BN)
    int k_blocks;              // ceil(K / 64)
    int group_m;               // rasterisation: tiles_m are walked in groups of this many
    int a_off_mn, a_off_k;     // coordinate offsets of the A operand inside its tensor map
    int b_off_mn, b_off_k;     // same for B
};

__device__ __forceinline__ void tile_coords(int tile, const GemmShape &s, int &m_blk, int &n_blk) {
    const int per_group = s.group_m * s.tiles_n;
    const int g = tile / per_group;
    const int first_m = g * s.group_m;
    const int gsz = min(s.tiles_m - first_m, s.group_m);
    const int r = tile - g * per_group;
    m_blk = first_m + r % gsz;
    n_blk = r / gsz;
}

// --------------------------------------------------------------------------
// bf16 helpers for the epilogues
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// store 8 consecutive values as bf16 (16 bytes, aligned)
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16 *p, const float *v) {
    uint4 u;
    u.x = pack_bf16x2(v[0], v[1]);
    u.y = pack_bf16x2(v[2], v[3]);
    u.z = pack_bf16x2(v[4], v[5]);
    u.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4 *>(p) = u;
}

__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16 *p, float *v) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}

// GeLU(u) = u Phi(u), Phi(u) = (1 + erf(u / sqrt 2)) / 2
__device__ __forceinline__ float gelu_f(float u) {
    return 0.5f * u * (1.0f + erff(u * 0.70710678118654752440f));
}
// GeLU'(u) = Phi(u) + u phi(u), phi(u) = exp(-u^2 / 2) / sqrt(2 pi)
__device__ __forceinline__ float gelu_grad_f(float u) {
    const float Phi = 0.5f * (1.0f + erff(u * 0.70710678118654752440f));
    const float phi = 0.39894228040143267794f * __expf(-0.5f * u * u);
    return Phi + u * phi;
}

// --------------------------------------------------------------------------
// Epilogues. `apply` runs in each of the 128 epilogue threads for one tile:
// `row` is the thread's global output row, `n0` the tile's first output
// column, `taddr` the TMEM address of the thread's warp quarter of the
// accumulator. Every thread of a warp executes the TMEM loads (they are
// warp-collective); only rows < M and columns < N are stored.
// --------------------------------------------------------------------------

// GEMM1 epilogue: U = acc + bA, Y = GeLU(U); both stored bf16.
struct EpiBiasGelu {
    struct Params {
        __nv_bfloat16 *U;
        __nv_bfloat16 *Y;
        const float *bias;  // [N] or null
        int64_t ld;
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int nc = n0 + c * 32;
            if (row >= s.M || nc >= s.N) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = nc + q * 8;
                if (n >= s.N) break;
                float u[8], y[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) u[i] = v[q * 8 + i] + (p.bias ? __ldg(p.bias + n + i) : 0.0f);
#pragma unroll
                for (int i = 0; i < 8; ++i) y[i] = gelu_f(u[i]);
                store_bf16x8(p.U + static_cast<int64_t>(row) * p.ld + n, u);
                store_bf16x8(p.Y + static_cast<int64_t>(row) * p.ld + n, y);
            }
        }
    }
};

// Plain epilogue: out = acc (+ bias), bf16.
struct EpiStore {
    struct Params {
        __nv_bfloat16 *out;
        const float *bias;  // [N] or null
        int64_t ld;
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int nc = n0 + c * 32;
            if (row >= s.M || nc >= s.N) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = nc + q * 8;
                if (n >= s.N) break;
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = v[q * 8 + i] + (p.bias ? __ldg(p.bias + n + i) : 0.0f);
                store_bf16x8(p.out + static_cast<int64_t>(row) * p.ld + n, o);
            }
        }
    }
};

// dY epilogue of the backward: dU = acc (.) GeLU'(U), U read from the saved activations.
struct EpiGeluGrad {
    struct Params {
        __nv_bfloat16 *dU;
        const __nv_bfloat16 *U;
        int64_t ld;
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int nc = n0 + c * 32;
            if (row >= s.M || nc >= s.N) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = nc + q * 8;
                if (n >= s.N) break;
                float u[8], d[8];
                load_bf16x8(p.U + static_cast<int64_t>(row) * p.ld + n, u);
#pragma unroll
                for (int i = 0; i < 8; ++i) d[i] = v[q * 8 + i] * gelu_grad_f(u[i]);
                store_bf16x8(p.dU + static_cast<int64_t>(row) * p.ld + n, d);
            }
        }
    }
};

// CE pass 1: logits of one vocabulary tile, reduced per token to (max, sum of
// exp(l - max)) over the real ids, plus the target logit where the target
// falls in this tile. The logits never leave the registers.
struct EpiCeStats {
    struct Params {
        float2 *stats;          // [n_tiles_total][T]: (max, sumexp) per tile and token
        float *tau;             // [T] target logit
        const int32_t *targets; // [T]
        int64_t T;
        int v_valid;
        int n_base;             // vocabulary id of GEMM column 0
        int tile_base;          // global tile index of GEMM tile column 0
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
        const bool live = row < s.M;
        const int tgt = live ? __ldg(p.targets + row) : -1;
        float m = -INFINITY, sum = 0.0f, tau = 0.0f;
        bool has_tau = false;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int g0 = p.n_base + n0 + c * 32;   // vocabulary id of v[0]
            const int nvalid = min(32, p.v_valid - g0);  // ids < v_valid are real
            if (nvalid > 0) {
                float cm = -INFINITY;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < nvalid) cm = fmaxf(cm, v[i]);
                const float nm = fmaxf(m, cm);
                float acc = sum * __expf(m - nm);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < nvalid) acc += __expf(v[i] - nm);
                sum = acc;
                m = nm;
            }
            const int tl = tgt - g0;
            if (tl >= 0 && tl < 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i == tl) tau = v[i];
                has_tau = true;
            }
        }
        if (live) {
            const int tile = p.tile_base + n0 / BN;
            p.stats[static_cast<int64_t>(tile) * p.T + row] = make_float2(m, sum);
            if (has_tau) p.tau[row] = tau;
        }
    }
};

// CE pass 2, first GEMM: recomputed logits -> dl = g (exp(l - lse) - onehot),
// zero on padded ids, stored bf16 into the chunk scratch.
struct EpiCeDlogits {
    struct Params {
        __nv_bfloat16 *dl;      // [T][ld] chunk scratch
        int64_t ld;
        const float *lse;       // [T]
        const int32_t *targets; // [T]
        float grad_scale;
        int v_valid;
        int n_base;             // vocabulary id of GEMM column 0
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
        const bool live = row < s.M;
        const float L = live ? __ldg(p.lse + row) : 0.0f;
        const int tgt = live ? __ldg(p.targets + row) : -1;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int nc = n0 + c * 32;
            if (!live || nc >= s.N) continue;
            const int g0 = p.n_base + nc;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = nc + q * 8;
                if (n >= s.N) break;
                float d[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int g = g0 + q * 8 + i;
                    const float pr = __expf(v[q * 8 + i] - L);
                    d[i] = g < p.v_valid ? p.grad_scale * (pr - (g == tgt ? 1.0f : 0.0f)) : 0.0f;
                }
                store_bf16x8(p.dl + static_cast<int64_t>(row) * p.ld + n, d);
            }
        }
    }
};

// fp32 accumulation across launches (dH summed over vocabulary chunks):
// mode 0: acc = v; 1: acc += v; 2: out = bf16(acc + v); 3: out = bf16(v).
struct EpiAccF32 {
    struct Params {
        float *acc;             // [M][ld] fp32
        __nv_bfloat16 *out;     // [M][ld] bf16
        int64_t ld;
        int mode;
    };
    template <int BN>
    __device__ static void apply(const Params &p, const GemmShape &s, int row, int n0, uint32_t taddr) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            ptx::tmem_ld32(taddr + c * 32, v);
            const int nc = n0 + c * 32;
            if (row >= s.M || nc >= s.N) continue;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int n = nc + q * 8;
                if (n >= s.N) break;
                const int64_t off = static_cast<int64_t>(row) * p.ld + n;
                float o[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) o[i] = v[q * 8 + i];
                if (p.mode == 1 || p.mode == 2) {
                    const float4 a0 = *reinterpret_cast<const float4 *>(p.acc + off);
                    const float4 a1 = *reinterpret_cast<const float4 *>(p.acc + off + 4);
                    o[0] += a0.x; o[1] += a0.y; o[2] += a0.z; o[3] += a0.w;
                    o[4] += a1.x; o[5] += a1.y; o[6] += a1.z; o[7] += a1.w;
                }
                if (p.mode <= 1) {
                    *reinterpret_cast<float4 *>(p.acc + off) = make_float4(o[0], o[1], o[2], o[3]);
                    *reinterpret_cast<float4 *>(p.acc + off + 4) = make_float4(o[4], o[5], o[6], o[7]);
                } else {
                    store_bf16x8(p.out + off, o);
                }
            }
        }
    }
};

// --------------------------------------------------------------------------
// The kernel
// --------------------------------------------------------------------------
template <int BN, bool A_MN, bool B_MN, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const GemmShape shp, const typename Epi::Params ep, uint32_t *err) {
    using C = TileCfg<BN>;
    constexpr int S = C::kStages;
    constexpr uint32_t kIdesc = ptx::idesc_bf16(kBM, BN, A_MN, B_MN);

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + S * C::kStageBytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            ptx::mbar_init(&full[i], 1);
            ptx::mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&tfull[i], 1);
            ptx::mbar_init(&tempty[i], 4);
        }
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(tmem_slot, C::kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int num_tiles = shp.tiles_m * shp.tiles_n;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;  // bit s: stage s has a load in flight or landed
            uint32_t issued_parity = 0;
            for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, shp, mb, nb);
                const int m0 = mb * kBM, n0 = nb * BN;
                for (int kb = 0; kb < shp.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, 1)) break;
                    ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    uint8_t *sa = smem + stage * C::kStageBytes;
                    uint8_t *sb = sa + C::kABytes;
                    const int k0 = kb * kBK;
                    if (!A_MN) {
                        ptx::tma_load_2d(sa, &tmA, &full[stage], k0 + shp.a_off_k, m0 + shp.a_off_mn);
                    } else {
#pragma unroll
                        for (int j = 0; j < kBM / 64; ++j)
                            ptx::tma_load_2d(sa + j * kMnBlockBytes, &tmA, &full[stage],
                                             m0 + shp.a_off_mn + 64 * j, k0 + shp.a_off_k);
                    }
                    if (!B_MN) {
                        ptx::tma_load_2d(sb, &tmB, &full[stage], k0 + shp.b_off_k, n0 + shp.b_off_mn);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            ptx::tma_load_2d(sb + j * kMnBlockBytes, &tmB, &full[stage],
                                             n0 + shp.b_off_mn + 64 * j, k0 + shp.b_off_k);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (*abort_flag) {
                // let every load this thread issued land before the CTA exits
                for (int s = 0; s < S; ++s)
                    if (issued & (1u << s)) ptx::mbar_wait_drain(&full[s], (issued_parity >> s) & 1u);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
                if (!ptx::mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, err, 2)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                bool ok = true;
                for (int kb = 0; kb < shp.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&full[stage], phase, abort_flag, err, 3)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint32_t sa = ptx::smem_u32(smem + stage * C::kStageBytes);
                    const uint32_t sb = sa + C::kABytes;
#pragma unroll
                    for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                        const uint64_t ad = A_MN ? ptx::sdesc_sw128(sa + kk * (kUmmaK * 128), kMnBlockBytes, 1024)
                                                 : ptx::sdesc_sw128(sa + kk * (kUmmaK * 2), 16, 1024);
                        const uint64_t bd = B_MN ? ptx::sdesc_sw128(sb + kk * (kUmmaK * 128), kMnBlockBytes, 1024)
                                                 : ptx::sdesc_sw128(sb + kk * (kUmmaK * 2), 16, 1024);
                        ptx::mma_bf16(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
                    }
                    ptx::mma_commit(&empty[stage]);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                ptx::mma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1;
            }
            // every MMA issued by this thread has completed once `drain` flips
            ptx::mma_commit(drain);
            ptx::mbar_wait_drain(drain, 0);
        }
    } else {
        // ------------------------------------------------ epilogue warps
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const int row_in_tile = quarter * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, shp, mb, nb);
            // the decision to go on must be warp-uniform: the TMEM loads are warp-collective
            const bool ok = ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            Epi::template apply<BN>(ep, shp, mb * kBM + row_in_tile, nb * BN, taddr);
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

}  // namespace
}  // namespace tpce
