// gemm.cuh -- the tensor-core GEMM behind every contraction of the block.
//
// D[M, N] = sum_k A[m, k] B[k, n] with an fp32 accumulator in tensor memory,
// followed by a fused epilogue. Operands are bf16 (tcgen05.mma kind::f16) or
// fp32 read as tf32 (kind::tf32). One persistent CTA per SM walks the output
// tiles; inside a CTA the work is split by warp:
//
//   warp 0      TMA producer: streams 128-row A and BN-row B tiles, 128 bytes
//               of K per row, into a ring of shared-memory stages (128-byte
//               swizzle).
//   warp 1      MMA issuer: one thread issues tcgen05.mma (M=128, N=BN) into
//               one of two TMEM accumulators; the warp owns the TMEM allocation.
//   warps 2..5  epilogue: tcgen05.ld the accumulator (one row per thread),
//               apply the fused epilogue, stage each 32x32 output chunk in
//               swizzled shared memory and write it with a TMA bulk tensor
//               store (or reduce-add), then hand the accumulator back, so the
//               next tile's MMAs overlap this tile's epilogue.
//
// bf16 operands can be K-major (the contraction dimension contiguous) or
// MN-major (the output dimension contiguous): the transposed operands of the
// backward GEMMs (Y^T dZ, X^T dU, dl^T H) can be read in place. An MN-major A
// costs the tensor core about 11%, so at large widths the callers give these
// GEMMs a K-major copy of A instead (made by a transpose pass, or for dl^T
// stored by the dl GEMM's own epilogue). tf32 operands are K-major.
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
#include <type_traits>

#include "ptx.cuh"

namespace tpce {
// Internal linkage: every translation unit gets its own kernels and launch
// state (a kernel instantiated in two units is two device functions).
namespace {

// Epilogue warps of the heavy epilogues (4: one per TMEM lane quarter; 8: two
// per quarter, splitting the columns). Build-time tuning knob.
#ifndef TPCE_EPI_WARPS
#define TPCE_EPI_WARPS 4
#endif
constexpr int kHeavyEpiWarps = TPCE_EPI_WARPS;

constexpr int kBM = 128;                 // tile rows (TMEM lanes)
constexpr uint32_t kRowBytes = 128;      // K bytes per smem row = one 128-byte swizzle span
constexpr uint32_t kMnBlockBytes = 64 * kRowBytes;  // one 64-wide MN block of a bf16 MN-major tile (64 K rows)

template <typename ElemT>
struct ElemTraits;
template <>
struct ElemTraits<__nv_bfloat16> {
    static constexpr int kBK = 64;       // elements of K per stage
    static constexpr int kUmmaK = 16;    // K of one tcgen05.mma kind::f16
    static constexpr uint32_t kFmt = 1;  // bf16
};
template <>
struct ElemTraits<float> {
    static constexpr int kBK = 32;
    static constexpr int kUmmaK = 8;     // K of one tcgen05.mma kind::tf32
    static constexpr uint32_t kFmt = 2;  // tf32
};

// Problem description shared by every role of the kernel.
struct GemmShape {
    int M, N, K;               // output rows, output columns, contraction length
    int tiles_m, tiles_n;      // ceil(M / 128), ceil(N / BN)
    int k_blocks;              // ceil(K / BK)
    int group_m;               // rasterisation: tiles_m are walked in groups of this many
    // Runs (CTA-pair kernel): a work unit is run_len consecutive column tiles
    // of one row-block, walked in order, the epilogue's row state carried
    // from tile to tile; unit_cols = tiles_n / run_len units per row-block.
    int run_len;
    int unit_cols;
    int a_off_mn, a_off_k;     // coordinate offsets of the A operand inside its tensor map
    int b_off_mn, b_off_k;     // same for B
    int b_gate_off;            // gated tiles: B column (or row) offset of the second half, else 0
    // Split tail (CTA-pair kernel): the first full_units work units are whole
    // tiles; each of the last tail_tiles tiles is split along K into `split`
    // units whose fp32 partials meet in `partial`, counted by `tickets`.
    int full_units;            // whole-tile units (all tiles when the tail is not split)
    int split;                 // K parts per tail tile (1: no split)
    int tail_tiles;            // tiles split
    float *partial;            // [tail_tiles * split][2 CTAs][128 rows][BN] fp32
    uint32_t *tickets;         // [tail_tiles][2 CTAs], zero at launch
    // L2 eviction priorities of the operand loads (CTA-pair kernel): 0 none;
    // 1 A's lines evict_last and B's evict_first, for launches whose group of
    // A panels fits in L2 and is reused by every column block the group walks
    // while B streams through once per group.
    int l2_hint;
    // Failure-path test knob, 0 in every ordinary launch. 1 (CTA-pair kernel
    // only): cluster 0 arms the full barrier of its first k-block but loads
    // nothing into it, so the MMA thread's bounded wait on it runs out.
    int debug_withhold;
};

// Work unit u: its tile, its K-block range, and its part (-1: a whole tile).
__device__ __forceinline__ void unit_coords(int u, const GemmShape &s, int &tile, int &kb0, int &kb1, int &part) {
    if (u < s.full_units) {
        tile = u;
        kb0 = 0;
        kb1 = s.k_blocks;
        part = -1;
    } else {
        const int j = u - s.full_units;
        const int tl = j / s.split;
        part = j - tl * s.split;
        tile = s.full_units + tl;
        kb0 = part * s.k_blocks / s.split;
        kb1 = (part + 1) * s.k_blocks / s.split;
    }
}

// Row-block and unit column of work unit `tile` (the column block when run_len = 1).
__device__ __forceinline__ void tile_coords(int tile, const GemmShape &s, int &m_blk, int &n_blk) {
    const int per_group = s.group_m * s.unit_cols;
    const int g = tile / per_group;
    const int first_m = g * s.group_m;
    const int gsz = min(s.tiles_m - first_m, s.group_m);
    const int r = tile - g * per_group;
    m_blk = first_m + r % gsz;
    n_blk = r / gsz;
}

// --------------------------------------------------------------------------
// Sequence-chunked operands. With sequence parallelism the activations enter
// and leave the tensor-parallel region as t sequence chunks in t separate
// buffers (one per rank): the column-parallel GEMM reads the all-gathered
// input from them, the row-parallel GEMM's epilogue writes the shard-summed
// output into them. One role of a launch may be chunked: the A operand, the
// B operand or output map 0. Its rows (the outer coordinate of its tensor
// map: M or K for an operand, M for the output) are split into chunks of
// `rows` rows, each with its own tensor map; a 128-row box never straddles
// two chunks because `rows` is a multiple of 128.
// --------------------------------------------------------------------------
constexpr int kMaxChunks = 16;
enum : int { kChunkNone = 0, kChunkA = 1, kChunkB = 2, kChunkC = 3 };

template <int kChunk>
struct ChunkSet {
    CUtensorMap m[kChunk != kChunkNone ? kMaxChunks : 1];
    int rows;   // rows per chunk
    int count;  // chunks in use
};

// Chunk c's map, picked by a switch so that every address handed to TMA is a
// fixed offset into the kernel parameter.
template <int kChunk>
__device__ __forceinline__ const CUtensorMap *chunk_map_at(const ChunkSet<kChunk> &cs, int c) {
    static_assert(kChunk == kChunkNone || kMaxChunks == 16, "the switch below lists 16 chunks");
    if constexpr (kChunk == kChunkNone) {
        return &cs.m[0];
    } else {
        switch (c) {
            case 1: return &cs.m[1];
            case 2: return &cs.m[2];
            case 3: return &cs.m[3];
            case 4: return &cs.m[4];
            case 5: return &cs.m[5];
            case 6: return &cs.m[6];
            case 7: return &cs.m[7];
            case 8: return &cs.m[8];
            case 9: return &cs.m[9];
            case 10: return &cs.m[10];
            case 11: return &cs.m[11];
            case 12: return &cs.m[12];
            case 13: return &cs.m[13];
            case 14: return &cs.m[14];
            case 15: return &cs.m[15];
            default: return &cs.m[0];
        }
    }
}

// The map holding outer coordinate y, and y rebased into that chunk. Rows
// past the last chunk stay in it (past its end: TMA fills them with zeros).
template <int kChunk>
__device__ __forceinline__ const CUtensorMap *chunk_map(const ChunkSet<kChunk> &cs, int &y) {
    int c = y / cs.rows;
    c = c < cs.count - 1 ? c : cs.count - 1;
    y -= c * cs.rows;
    return chunk_map_at(cs, c);
}

// The chunk an operand's loads are in, kept across the K loop so that the
// producer never divides or switches per k-block: K-major operands (outer
// coordinate M or N) pick their chunk once per tile; MN-major ones (outer
// coordinate K) step `dy` rows per k-block and change map only at a chunk
// boundary (dy divides the chunk rows).
template <int kChunk>
struct ChunkCursor {
    const CUtensorMap *map;
    int y;  // outer coordinate inside the current chunk
    int c;  // current chunk
    __device__ __forceinline__ void init(const ChunkSet<kChunk> &cs, int y0) {
        c = y0 / cs.rows;
        c = c < cs.count - 1 ? c : cs.count - 1;
        y = y0 - c * cs.rows;
        map = chunk_map_at(cs, c);
    }
    __device__ __forceinline__ void advance(const ChunkSet<kChunk> &cs, int dy) {
        y += dy;
        if (y >= cs.rows && c < cs.count - 1) {
            y -= cs.rows;
            ++c;
            map = chunk_map_at(cs, c);
        }
    }
};

// Bring every chunk's descriptor into the TMA descriptor cache up front
// (switching maps mid-tile otherwise stalls on descriptor fetches).
template <int kChunk>
__device__ __forceinline__ void prefetch_chunk_maps(const ChunkSet<kChunk> &cs) {
    if constexpr (kChunk != kChunkNone) {
        for (int c = 0; c < cs.count; ++c) ptx::prefetch_tmap(chunk_map_at(cs, c));
    }
}

// --------------------------------------------------------------------------
// 8-element loads for the epilogues (16- or 32-byte aligned)
// --------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float *v) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void load8(const float *p, float *v) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// 32 bias values starting at column n (zeros where absent); N % 8 == 0, so
// every 8-column group is entirely inside or outside [0, N).
__device__ __forceinline__ void load_bias32(const float *bias, int n, int N, float *b) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (bias && n + 8 * q < N) {
            load8(bias + n + 8 * q, b + 8 * q);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) b[8 * q + i] = 0.0f;
        }
    }
}

// Standard normal CDF Phi(u) = (1 + erf(u / sqrt 2)) / 2, with erf taken from
// Abramowitz & Stegun, Handbook of Mathematical Functions, formula 7.1.26:
// for z >= 0, erf(z) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) e^{-z^2},
// t = 1 / (1 + p z), |error| <= 1.5e-7. With z = |u| / sqrt 2 the factor
// e^{-z^2} = e^{-u^2 / 2} is also the Gaussian density's exponent, so GeLU'
// reuses it. `g` receives e^{-u^2 / 2}.
__device__ __forceinline__ float normal_cdf(float u, float &g) {
    constexpr float p = 0.3275911f;
    constexpr float a1 = 0.254829592f, a2 = -0.284496736f, a3 = 1.421413741f, a4 = -1.453152027f,
                    a5 = 1.061405429f;
    const float z = fabsf(u) * 0.70710678118654752440f;
    const float t = __fdividef(1.0f, fmaf(p, z, 1.0f));
    g = __expf(-0.5f * u * u);
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, a5, a4), a3), a2), a1);
    const float erf_z = 1.0f - poly * g;  // erf(|u| / sqrt 2)
    return 0.5f + 0.5f * copysignf(erf_z, u);
}
// GeLU(u) = u Phi(u)
__device__ __forceinline__ float gelu_f(float u) {
    float g;
    return u * normal_cdf(u, g);
}
// GeLU'(u) = Phi(u) + u phi(u), phi(u) = e^{-u^2 / 2} / sqrt(2 pi)
__device__ __forceinline__ float gelu_grad_f(float u) {
    float g;
    const float Phi = normal_cdf(u, g);
    return fmaf(u * 0.39894228040143267794f, g, Phi);
}

// Swish(x) = x sigmoid(x), sigmoid(x) = 1 / (1 + e^{-x}); for x << 0 the
// exponential overflows to +inf and the quotient to 0, the right limit.
__device__ __forceinline__ float sigmoid_f(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }

// --------------------------------------------------------------------------
// Output staging. An epilogue warp writes each 32-row x 32-column chunk of an
// output into a shared-memory buffer, one row per lane, swizzled exactly as
// the TMA store of that buffer expects (bf16: 64-byte rows, 64-byte swizzle;
// fp32: 128-byte rows, 128-byte swizzle); one lane then stores the chunk with
// a TMA bulk tensor store, which writes whole lines, clips the tensor's ragged
// edges and runs asynchronously.
// --------------------------------------------------------------------------
template <typename OutT>
struct Stage;
template <>
struct Stage<__nv_bfloat16> {
    static constexpr uint32_t kBytes = 32 * 64;
    static constexpr int kSwizzle = 64;
    // 16-byte piece j of row r lives at piece j ^ ((r >> 1) & 3)
    __device__ static void write(uint8_t *buf, int r, const float *v) {
        uint8_t *row = buf + r * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 u;
            u.x = pack_bf16x2(v[8 * j + 0], v[8 * j + 1]);
            u.y = pack_bf16x2(v[8 * j + 2], v[8 * j + 3]);
            u.z = pack_bf16x2(v[8 * j + 4], v[8 * j + 5]);
            u.w = pack_bf16x2(v[8 * j + 6], v[8 * j + 7]);
            *reinterpret_cast<uint4 *>(row + ((j ^ ((r >> 1) & 3)) << 4)) = u;
        }
    }
    __device__ static void read(const uint8_t *buf, int r, float *v) {
        const uint8_t *row = buf + r * 64;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint4 u = *reinterpret_cast<const uint4 *>(row + ((j ^ ((r >> 1) & 3)) << 4));
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float2 f = __bfloat1622float2(h[i]);
                v[8 * j + 2 * i] = f.x;
                v[8 * j + 2 * i + 1] = f.y;
            }
        }
    }
};
// The same 32 x 32 bf16 chunk staged transposed, for a TMA store into the
// transposed output (rows: the chunk's columns, columns: its rows): lane r
// writes its row's 32 values down column r. Element (c, r) of the staged box
// lives in row c, 16-byte piece (r / 8) ^ ((c >> 1) & 3), slot r % 8; for
// each c the warp's 32 two-byte writes fill one 64-byte row.
struct StageT {
    __device__ static void write(uint8_t *buf, int r, const float *v) {
        const int piece = r >> 3, slot = (r & 7) * 2;
#pragma unroll
        for (int c = 0; c < 32; ++c)
            *reinterpret_cast<__nv_bfloat16 *>(buf + c * 64 + ((piece ^ ((c >> 1) & 3)) << 4) + slot) =
                __float2bfloat16_rn(v[c]);
    }
};
template <>
struct Stage<float> {
    static constexpr uint32_t kBytes = 32 * 128;
    static constexpr int kSwizzle = 128;
    // 16-byte piece j of row r lives at piece j ^ (r & 7)
    __device__ static void write(uint8_t *buf, int r, const float *v) {
        uint8_t *row = buf + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4 *>(row + ((j ^ (r & 7)) << 4)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    __device__ static void read(const uint8_t *buf, int r, float *v) {
        const uint8_t *row = buf + r * 128;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float4 f = *reinterpret_cast<const float4 *>(row + ((j ^ (r & 7)) << 4));
            v[4 * j] = f.x;
            v[4 * j + 1] = f.y;
            v[4 * j + 2] = f.z;
            v[4 * j + 3] = f.w;
        }
    }
};

// --------------------------------------------------------------------------
// Epilogues. Each turns the fp32 accumulator values of one 32-column chunk of
// the thread's output row into kOuts output chunks (stored by the kernel), or
// reduces them itself (kOuts = 0). An epilogue with kIns = 1 or 2 also
// receives, in in[0 .. kIns), the matching 32 values of kIns inputs of the
// output's shape, which the kernel brings into shared memory with TMA loads
// one chunk ahead. begin/end run once per tile and row. `live` is false for
// rows >= M or chunks at columns >= N: such values are never stored, and the
// epilogue must not read memory for them.
//
// Where the outputs and inputs go (defaults in EpiBase):
//   out_map(k)     which of the kernel's two output tensor maps output k uses;
//   out_col(p, k)  column offset of output k inside that map;
//   in_col(p, i)   column offset of input i inside the input map.
// A gated epilogue (kGated) runs on tiles whose accumulator holds two halves,
// [gate | up], each of the same output columns: the B tile's first half comes
// from B's columns n.., the second from n + b_gate_off... The epilogue sees
// the gate half in v and the up half in in[0]; a tile spans half as many
// output columns as accumulator columns.
// --------------------------------------------------------------------------
struct NoRow {};

struct EpiBase {
    static constexpr bool kGated = false;
    // output 1 is the transpose of output 0's tile ([N, M], bf16): staged by
    // StageT and stored at (row, column) = (n, m)
    static constexpr bool kTransOut1 = false;
    __host__ __device__ static constexpr int out_map(int k) { return k; }
    template <class P>
    __device__ static int out_col(const P &, int) { return 0; }
    template <class P>
    __device__ static int in_col(const P &, int) { return 0; }
};

// Number of distinct output tensor maps an epilogue stores through.
template <class Epi>
constexpr int num_out_maps() {
    int m = 0;
    for (int k = 0; k < Epi::kOuts; ++k) m = Epi::out_map(k) + 1 > m ? Epi::out_map(k) + 1 : m;
    return m;
}

// GEMM1 epilogue: U = acc + bA, Y = GeLU(U).
template <typename OutT>
struct EpiBiasGelu : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 2;
    static constexpr int kIns = 0;
    using Out = OutT;
    using Row = NoRow;
    struct Params {
        const float *bias;  // [N] or null
    };
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &p, Row &, int, int n, int N, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
        float b[32];
        load_bias32(p.bias, n, N, b);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            o[0][i] = v[i] + b[i];
            o[1][i] = gelu_f(o[0][i]);
        }
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// Plain epilogue: out = acc (+ bias).
template <typename OutT>
struct EpiStore : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 1;
    static constexpr int kIns = 0;
    using Out = OutT;
    using Row = NoRow;
    struct Params {
        const float *bias;  // [N] or null
    };
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &p, Row &, int, int n, int N, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
        float b[32];
        load_bias32(p.bias, n, N, b);
#pragma unroll
        for (int i = 0; i < 32; ++i) o[0][i] = v[i] + b[i];
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// dY epilogue of the backward: dU = acc (.) GeLU'(U); the saved U arrives as
// the kernel-loaded input chunk.
template <typename OutT>
struct EpiGeluGrad : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 1;
    static constexpr int kIns = 1;
    using Out = OutT;
    using Row = NoRow;
    struct Params {};
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &, Row &, int, int, int, bool, float (&v)[32], const float (&u)[2][32],
                                 float (&o)[kOuts][32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[0][i] = v[i] * gelu_grad_f(u[0][i]);
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// SwiGLU forward (gated tile): G = acc_gate + b_gate, Up = acc_up + b_up,
// Y = Swish(G) Up. Outputs: G and Up into the [T, 2f] map at columns n and
// f_off + n, Y into the [T, f] map.
template <typename OutT>
struct EpiSwiGlu : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 3;
    static constexpr int kIns = 0;
    static constexpr bool kGated = true;
    using Out = OutT;
    using Row = NoRow;
    struct Params {
        const float *bias;  // [2 f_off] (gate biases, then up biases) or null
        int f_off;          // f: column offset of the up half in W1, the bias and GU
    };
    __host__ __device__ static constexpr int out_map(int k) { return k == 2 ? 1 : 0; }
    __device__ static int out_col(const Params &p, int k) { return k == 1 ? p.f_off : 0; }
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &p, Row &, int, int n, int N, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
        float bg[32], bu[32];
        load_bias32(p.bias, n, N, bg);
        load_bias32(p.bias ? p.bias + p.f_off : nullptr, n, N, bu);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float g = v[i] + bg[i];
            const float u = in[0][i] + bu[i];
            o[0][i] = g;
            o[1][i] = u;
            o[2][i] = g * sigmoid_f(g) * u;
        }
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// SwiGLU dY epilogue of the backward: with dY = acc and the saved G, Up as the
// two inputs, dG = dY Up Swish'(G), dUp = dY Swish(G), where
// Swish'(g) = s (1 + g (1 - s)), s = sigmoid(g). Outputs into the [T, 2f] map
// at columns n and f_off + n.
template <typename OutT>
struct EpiSwiGluGrad : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 2;
    static constexpr int kIns = 2;
    using Out = OutT;
    using Row = NoRow;
    struct Params {
        int f_off;  // f: column offset of the up half in GU and dGU
    };
    __host__ __device__ static constexpr int out_map(int) { return 0; }
    __device__ static int out_col(const Params &p, int k) { return k == 1 ? p.f_off : 0; }
    __device__ static int in_col(const Params &p, int i) { return i == 1 ? p.f_off : 0; }
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &, Row &, int, int, int, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const float g = in[0][i], u = in[1][i];
            const float s = sigmoid_f(g);
            o[0][i] = v[i] * u * (s * fmaf(g, 1.0f - s, 1.0f));
            o[1][i] = v[i] * (g * s);
        }
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// CE pass 1: logits of a run of vocabulary tiles (one tile on the one-CTA
// kernel), reduced per token to (max, sum of exp(l - max)) over the real ids,
// plus the target logit where the target falls in the run. The running
// (max, sum) is carried from tile to tile of the run in registers. The logits
// never leave the registers. One warp per TMEM lane quarter, so each thread
// sees its token's whole tile row.
//
// A shard covered by one run stores its (max, sum) straight into the shard's
// statistics. A shard cut into several runs ("parts") stores each part's pair;
// then, per 32-row slab, the warp that finishes the shard's last part -- known
// from an atomic ticket per (slab, shard), with no waiting -- folds the parts
// in part order into the shard's pair. Either way the exchange across shards
// sees exactly one (max, sum) per shard and token.
struct EpiCeStats : EpiBase {
    static constexpr int kWarps = 4;
    static constexpr int kOuts = 0;
    static constexpr int kIns = 0;
    using Out = float;
    struct Row {
        int tgt;
        float m, sum, tau;
        bool has_tau;
    };
    struct Params {
        float2 *stats;          // [t][T]: each shard's (max, sumexp) per token
        float2 *parts;          // [t * parts_per_shard][T]: the parts' pairs (unused with one part per shard)
        uint32_t *tickets;      // [ceil(T / 32)][t]: parts finished per slab and shard, zero at launch
        float *tau;             // [T] target logit
        const int32_t *targets; // [T]
        int64_t T;
        int v_valid;
        int n_base;             // vocabulary id of GEMM column 0
        int tile_base;          // global part index of GEMM tile column 0
        int bn;                 // tile width
        int run_len;            // tiles per part: a part is one work unit's run of tiles
        int parts_per_shard;
        int shards;             // t
    };
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &p, int row, bool live) {
        return Row{live ? __ldg(p.targets + row) : -1, -INFINITY, 0.0f, 0.0f, false};
    }
    __device__ static void chunk(const Params &p, Row &r, int, int n, int, bool, float (&v)[32],
                                 const float (&)[2][32], float (&)[1][32]) {
        const int g0 = p.n_base + n;                 // vocabulary id of v[0]
        const int nvalid = min(32, p.v_valid - g0);  // ids < v_valid are real
        if (nvalid == 32) {
            float cm = v[0];
#pragma unroll
            for (int i = 1; i < 32; ++i) cm = fmaxf(cm, v[i]);
            const float nm = fmaxf(r.m, cm);
            float acc = r.sum * __expf(r.m - nm);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc += __expf(v[i] - nm);
            r.sum = acc;
            r.m = nm;
        } else if (nvalid > 0) {  // the chunk that holds the last real ids
            float cm = -INFINITY;
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nvalid) cm = fmaxf(cm, v[i]);
            const float nm = fmaxf(r.m, cm);
            float acc = r.sum * __expf(r.m - nm);
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < nvalid) acc += __expf(v[i] - nm);
            r.sum = acc;
            r.m = nm;
        }
        const int tl = r.tgt - g0;
        if (tl >= 0 && tl < 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i == tl) r.tau = v[i];
            r.has_tau = true;
        }
    }
    // Called by all 32 lanes of a warp together, lane l on row row0 + l; n0 is
    // the first column of the run's last tile.
    __device__ static void end(const Params &p, Row &r, int row, int n0, bool live) {
        const int part = p.tile_base + (n0 / p.bn) / p.run_len;
        const int shard = part / p.parts_per_shard;
        if (r.has_tau) p.tau[row] = r.tau;
        if (p.parts_per_shard == 1) {
            if (live) p.stats[static_cast<int64_t>(shard) * p.T + row] = make_float2(r.m, r.sum);
            return;
        }
        if (live) p.parts[static_cast<int64_t>(part) * p.T + row] = make_float2(r.m, r.sum);
        const int lane = static_cast<int>(threadIdx.x & 31u);
        const int row0 = row - lane;
        if (row0 >= p.T) return;  // no real rows in this slab (the same for every part)
        __threadfence();          // this part's pairs are visible GPU-wide before the ticket
        __syncwarp();
        uint32_t *ticket = p.tickets + static_cast<int64_t>(row0 / 32) * p.shards + shard;
        uint32_t t = 0;
        if (lane == 0) t = atomicAdd(ticket, 1u);
        t = __shfl_sync(0xffffffffu, t, 0);
        if (t != static_cast<uint32_t>(p.parts_per_shard - 1)) return;  // another part folds
        __threadfence();  // every part's pairs are visible to this warp
        if (live) {
            // the fold of the combine: parts with no real id (sum 0) are skipped
            float m = -INFINITY, sum = 0.0f;
            const float2 *src = p.parts + static_cast<int64_t>(shard) * p.parts_per_shard * p.T + row;
            for (int k = 0; k < p.parts_per_shard; ++k) {
                const float2 q = __ldcg(src + static_cast<int64_t>(k) * p.T);  // written by other SMs
                if (q.y > 0.0f) {
                    const float nm = fmaxf(m, q.x);
                    sum = sum * expf(m - nm) + q.y * expf(q.x - nm);
                    m = nm;
                }
            }
            p.stats[static_cast<int64_t>(shard) * p.T + row] = make_float2(m, sum);
        }
        __syncwarp();
        if (lane == 0) *ticket = 0u;  // every part has counted: leave the ticket clear
    }
};

// CE pass 2, first GEMM: recomputed logits -> dl = g (exp(l - lse) - onehot),
// zero on padded ids. Per element only the exponential: for g > 0 the scale
// is folded into it (g exp(l - lse) = exp(l - (lse - ln g))); the padding and
// the target column are handled per 32-column chunk, in the rare chunks that
// hold them.
template <typename OutT>
struct EpiCeDlogits : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 1;
    static constexpr int kIns = 0;
    using Out = OutT;
    struct Row {
        float c;    // exp(l - c) * mul = g softmax(l)
        float mul;  // 1 when g > 0 (folded into c), else g
        int tgt;
    };
    struct Params {
        const float *lse;       // [T]
        const int32_t *targets; // [T]
        float grad_scale;
        int v_valid;
        int n_base;             // vocabulary id of GEMM column 0
    };
    __device__ static int mode(const Params &) { return 0; }
    __device__ static Row begin(const Params &p, int row, bool live) {
        const float lse = live ? __ldg(p.lse + row) : 0.0f;
        const bool fold = p.grad_scale > 0.0f;
        return Row{fold ? lse - logf(p.grad_scale) : lse, fold ? 1.0f : p.grad_scale,
                   live ? __ldg(p.targets + row) : -1};
    }
    __device__ static void chunk(const Params &p, Row &r, int, int n, int, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
        const int g0 = p.n_base + n;  // vocabulary id of v[0]
        if (r.mul == 1.0f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = __expf(v[i] - r.c);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[0][i] = r.mul * __expf(v[i] - r.c);
        }
        if (g0 + 32 > p.v_valid) {  // padded ids: zero gradient
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (g0 + i >= p.v_valid) o[0][i] = 0.0f;
        }
        const int tl = r.tgt - g0;
        if (static_cast<unsigned>(tl) < 32u) {  // the target column: minus g
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i == tl) o[0][i] -= p.grad_scale;
        }
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// The same dl tile stored twice: dl [T, vc] and its transpose dl^T [vc, T]
// (the K-major A operand of dE = dl^T H).
struct EpiCeDlogitsT : EpiCeDlogits<__nv_bfloat16> {
    using Base = EpiCeDlogits<__nv_bfloat16>;
    static constexpr int kOuts = 2;
    static constexpr bool kTransOut1 = true;
    // fills o[0]; the transposed output is staged from o[0] as well
    __device__ static void chunk(const Params &p, Row &r, int row, int n, int N, bool live, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
        Base::chunk(p, r, row, n, N, live, v, in, reinterpret_cast<float(&)[1][32]>(o));
    }
};

// fp32 output stored (mode 0) or added element-wise into global memory by the
// TMA reduction (mode 1): dH summed over vocabulary chunks, in chunk order.
struct EpiF32Accumulate : EpiBase {
    static constexpr int kWarps = kHeavyEpiWarps;
    static constexpr int kOuts = 1;
    static constexpr int kIns = 0;
    using Out = float;
    using Row = NoRow;
    struct Params {
        int add;  // 0: store, 1: add into the existing values
    };
    __device__ static int mode(const Params &p) { return p.add; }
    __device__ static Row begin(const Params &, int, bool) { return {}; }
    __device__ static void chunk(const Params &, Row &, int, int, int, bool, float (&v)[32],
                                 const float (&in)[2][32], float (&o)[kOuts][32]) {
#pragma unroll
        for (int i = 0; i < 32; ++i) o[0][i] = v[i];
    }
    __device__ static void end(const Params &, Row &, int, int, bool) {}
};

// --------------------------------------------------------------------------
// The epilogue driver shared by the one-CTA and the CTA-pair kernels.
// Per epilogue warp, shared memory holds 2 staging buffers per output and 2
// sets of kIns input buffers, each a 32 x 32 chunk; each input set has one
// mbarrier.
// --------------------------------------------------------------------------
template <class Epi>
struct EpiSmem {
    using OutT = typename Epi::Out;
    static constexpr uint32_t kChunkBytes = Stage<OutT>::kBytes;
    static constexpr uint32_t kOutBytes = Epi::kOuts * 2 * kChunkBytes;
    static constexpr uint32_t kInBytes = Epi::kIns * 2 * kChunkBytes;
    static constexpr uint32_t kWarpBytes = kOutBytes + kInBytes;
    static constexpr uint32_t kBytes = static_cast<uint32_t>(Epi::kWarps) * kWarpBytes;
};

struct EpiWarp {
    uint8_t *stage;     // this warp's buffers (outputs, then inputs)
    uint64_t *in_bar;   // this warp's two input barriers
    int chunk_ctr;      // output chunks staged so far
    bool prev_stored;   // whether the previous output chunk was stored
    uint32_t in_issued; // input chunk loads issued
    uint32_t in_used;   // input chunk loads consumed
};

// Start the TMA loads of the input chunks at (n + in_col(i), row0) into the
// next input set.
template <class Epi>
__device__ __forceinline__ void epi_issue_input(EpiWarp &w, const typename Epi::Params &ep, const CUtensorMap *tmIn,
                                                int lane, int n, int row0) {
    if constexpr (Epi::kIns > 0) {
        constexpr uint32_t kB = EpiSmem<Epi>::kChunkBytes;
        if (lane == 0) {
            const uint32_t b = w.in_issued & 1u;
            ptx::mbar_arrive_expect_tx(&w.in_bar[b], Epi::kIns * kB);
#pragma unroll
            for (int i = 0; i < Epi::kIns; ++i)
                ptx::tma_load_2d(w.stage + EpiSmem<Epi>::kOutBytes + (b * Epi::kIns + i) * kB, tmIn, &w.in_bar[b],
                                 n + Epi::in_col(ep, i), row0);
        }
        ++w.in_issued;
    }
}

// Land the input loads still in flight (abort path), within a bounded time.
template <class Epi>
__device__ __forceinline__ void epi_drain_inputs(EpiWarp &w) {
    if constexpr (Epi::kIns > 0) {
        while (w.in_used < w.in_issued) {
            ptx::mbar_wait_drain(&w.in_bar[w.in_used & 1u], (w.in_used >> 1) & 1u);
            ++w.in_used;
        }
    }
}

// Where an epilogue reads the accumulator from: tensor memory (one row per
// thread, warp-collective loads), or -- for a split tail tile -- the sum of
// the fp32 partials of its K parts, added in part order so that the result
// does not depend on which part finished last.
struct TmemAcc {
    uint32_t taddr;  // this warp's lane quarter, column 0
    __device__ __forceinline__ void load(int col, float (&v)[32]) const { ptx::tmem_ld32(taddr + col, v); }
};
// A partial is stored column-major, element (row, col) at col * 128 + row,
// so that the 32 lanes of a warp (32 consecutive rows) touch one 128-byte
// line per column.
struct PartialAcc {
    const float *row;     // this thread's row of part 0 (element (row, 0))
    int64_t part_stride;  // floats between parts
    int parts;
    __device__ __forceinline__ void load(int col, float (&v)[32]) const {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
        for (int p = 0; p < parts; ++p) {
            const float *src = row + p * part_stride + static_cast<int64_t>(col) * kBM;
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += __ldcg(src + i * kBM);  // written by other SMs: not through L1
        }
    }
};

// One tile's epilogue for this warp: chunks [c0, c1) of its 32 rows starting
// at row0, columns from n0. The input chunk c0 must already be issued. Gated
// epilogues read the up half of chunk c at accumulator column up_col + 32 c.
// The row state rs is begun on the first tile of a run and ended on its last
// (both for a lone tile). Returns false if a bounded wait gave up.
template <class Epi, int kChunk, class Acc>
__device__ __forceinline__ bool epi_tile(const typename Epi::Params &ep, const GemmShape &shp, const Acc &acc,
                                         uint32_t up_col, int row0, int n0, int c0, int c1, int lane, EpiWarp &w,
                                         typename Epi::Row &rs, bool first, bool last,
                                         const CUtensorMap *tmC0, const CUtensorMap *tmC1,
                                         const CUtensorMap *tmIn, const ChunkSet<kChunk> *cs,
                                         volatile int *abort_flag, uint32_t *err) {
    using OutT = typename Epi::Out;
    constexpr int kOuts = Epi::kOuts;
    constexpr uint32_t kB = EpiSmem<Epi>::kChunkBytes;
    static_assert(Epi::kIns <= 2 && !(Epi::kGated && Epi::kIns > 0), "epilogue inputs");
    static_assert(!Epi::kTransOut1 || (Epi::kOuts == 2 && kChunk != kChunkC &&
                                       std::is_same<OutT, __nv_bfloat16>::value),
                  "a transposed second output: bf16, unchunked");
    const int row = row0 + lane;
    // output map 0 and the row coordinate in it (a sequence chunk, if chunked)
    const CUtensorMap *tm0 = tmC0;
    int y0 = row0;
    if constexpr (kChunk == kChunkC) tm0 = chunk_map(*cs, y0);
    if (first) rs = Epi::begin(ep, row, row < shp.M);
#pragma unroll 1
    for (int c = c0; c < c1; ++c) {
        const int n = n0 + c * 32;
        if (c + 1 < c1) epi_issue_input<Epi>(w, ep, tmIn, lane, n + 32, row0);
        float v[32];
        acc.load(c * 32, v);
        float in[2][32];
        if constexpr (Epi::kGated) acc.load(static_cast<int>(up_col) + c * 32, in[0]);
        if constexpr (Epi::kIns > 0) {
            const uint32_t b = w.in_used & 1u;
            const bool ok = ptx::mbar_wait(&w.in_bar[b], (w.in_used >> 1) & 1u, abort_flag, err, 5);
            if (!__all_sync(0xffffffffu, ok)) return false;
#pragma unroll
            for (int i = 0; i < Epi::kIns; ++i)
                Stage<OutT>::read(w.stage + EpiSmem<Epi>::kOutBytes + (b * Epi::kIns + i) * kB, lane, in[i]);
            __syncwarp();  // every lane has read the buffers before they are loaded again
            ++w.in_used;
        }
        const bool col_live = n < shp.N;
        float o[kOuts > 0 ? kOuts : 1][32];
        Epi::chunk(ep, rs, row, n, shp.N, row < shp.M && col_live, v, in, o);
        if constexpr (kOuts > 0) {
            const int buf = w.chunk_ctr & 1;
            // the buffer's previous store (two chunks ago) must have read it
            if (lane == 0) {
                if (w.prev_stored)
                    ptx::bulk_wait_read<1>();
                else
                    ptx::bulk_wait_read<0>();
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < kOuts; ++k) {
                if (Epi::kTransOut1 && k == 1)
                    StageT::write(w.stage + (2 * k + buf) * kB, lane, o[0]);
                else
                    Stage<OutT>::write(w.stage + (2 * k + buf) * kB, lane, o[k]);
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            const bool do_store = col_live && row0 < shp.M;
            if (lane == 0 && do_store) {
#pragma unroll
                for (int k = 0; k < kOuts; ++k) {
                    const uint8_t *src = w.stage + (2 * k + buf) * kB;
                    const CUtensorMap *tm = Epi::out_map(k) == 0 ? tm0 : tmC1;
                    const bool trans = Epi::kTransOut1 && k == 1;
                    const int col = trans ? row0 : n + Epi::out_col(ep, k);
                    const int y = trans ? n : (Epi::out_map(k) == 0 ? y0 : row0);
                    if (Epi::mode(ep) == 1)
                        ptx::tma_reduce_add_2d(tm, src, col, y);
                    else
                        ptx::tma_store_2d(tm, src, col, y);
                }
                ptx::bulk_commit();
            }
            w.prev_stored = do_store;
            ++w.chunk_ctr;
        }
    }
    if (last) Epi::end(ep, rs, row, n0, row < shp.M);
    return true;
}

// --------------------------------------------------------------------------
// Shared-memory plan of one instantiation: operand stages, then epilogue
// staging, then barriers.
// --------------------------------------------------------------------------
constexpr uint32_t kSmemMax = 232448;  // opt-in dynamic shared memory per block
constexpr uint32_t kBarrierBytes = 512;

template <int BN, class Epi>
struct KernelCfg {
    static_assert(BN == 128 || BN == 192 || BN == 256, "tile width");
    static constexpr uint32_t kABytes = kBM * kRowBytes;
    static constexpr uint32_t kBBytes = BN * kRowBytes;
    static constexpr uint32_t kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kStagingBytes = EpiSmem<Epi>::kBytes;
    static constexpr uint32_t kFree = kSmemMax - 1024 - kBarrierBytes - kStagingBytes;
    static constexpr int kStages = (kFree / kStageBytes) > 6 ? 6 : static_cast<int>(kFree / kStageBytes);
    static_assert(kStages >= 3, "too few pipeline stages");
    static constexpr uint32_t kTmemCols = BN == 128 ? 256 : 512;  // two accumulators, power of two
    static constexpr uint32_t kSmemBytes = kStages * kStageBytes + kStagingBytes + 1024 + kBarrierBytes;
};

// --------------------------------------------------------------------------
// The kernel
// --------------------------------------------------------------------------
template <typename ElemT, int BN, bool A_MN, bool B_MN, class Epi, int kChunk>
__global__ void __launch_bounds__(64 + 32 * Epi::kWarps, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
                   const __grid_constant__ CUtensorMap tmIn, const __grid_constant__ ChunkSet<kChunk> cs,
                   const GemmShape shp, const typename Epi::Params ep, uint32_t *err) {
    using C = KernelCfg<BN, Epi>;
    using ET = ElemTraits<ElemT>;
    using OutT = typename Epi::Out;
    static_assert(std::is_same<ElemT, __nv_bfloat16>::value || (!A_MN && !B_MN),
                  "tf32 operands are K-major");
    static_assert(Epi::kWarps == 4 || Epi::kWarps == 8, "epilogue warps");
    constexpr int S = C::kStages;
    constexpr int kBK = ET::kBK;
    constexpr int kUmmaK = ET::kUmmaK;
    constexpr uint32_t kIdesc = ptx::idesc_f32acc(kBM, BN, ET::kFmt, A_MN, B_MN);
    constexpr int kGroups = Epi::kWarps / 4;  // epilogue warps per TMEM lane quarter
    constexpr int kTileN = Epi::kGated ? BN / 2 : BN;  // output columns per tile
    constexpr int kChunks = kTileN / 32;
    constexpr int kOuts = Epi::kOuts;
    static_assert(!Epi::kGated || BN % 128 == 0, "gated tiles: halves of whole 64-wide blocks");
    static_assert(!(Epi::kGated && kChunk == kChunkB), "gated tiles read an unchunked B");

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *staging = smem + S * C::kStageBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(staging + C::kStagingBytes);
    uint64_t *empty = full + S;
    uint64_t *tfull = empty + S;
    uint64_t *tempty = tfull + 2;
    uint64_t *drain = tempty + 2;
    uint64_t *in_bars = drain + 1;  // 2 per epilogue warp
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(in_bars + 2 * Epi::kWarps);
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
            ptx::mbar_init(&tempty[i], Epi::kWarps);
        }
        for (int i = 0; i < 2 * Epi::kWarps; ++i) ptx::mbar_init(&in_bars[i], 1);
        ptx::mbar_init(drain, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if constexpr (kChunk == kChunkA || kChunk == kChunkB) prefetch_chunk_maps(cs);
    }
    if constexpr (kChunk == kChunkC) {
        if (warp == 2 && lane == 0) prefetch_chunk_maps(cs);
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
                const int m0 = mb * kBM, n0 = nb * kTileN;
                ChunkCursor<kChunk> cur;
                if constexpr (kChunk == kChunkA) cur.init(cs, A_MN ? shp.a_off_k : m0 + shp.a_off_mn);
                if constexpr (kChunk == kChunkB) cur.init(cs, B_MN ? shp.b_off_k : n0 + shp.b_off_mn);
                for (int kb = 0; kb < shp.k_blocks; ++kb) {
                    if (!ptx::mbar_wait(&empty[stage], phase ^ 1, abort_flag, err, 1)) break;
                    ptx::mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    uint8_t *sa = smem + stage * C::kStageBytes;
                    uint8_t *sb = sa + C::kABytes;
                    const int k0 = kb * kBK;
                    // A's outer coordinate: M (K-major) or K (MN-major)
                    int ya = A_MN ? k0 + shp.a_off_k : m0 + shp.a_off_mn;
                    const CUtensorMap *ma = &tmA;
                    if constexpr (kChunk == kChunkA) {
                        ma = cur.map;
                        ya = cur.y;
                    }
                    if (!A_MN) {
                        ptx::tma_load_2d(sa, ma, &full[stage], k0 + shp.a_off_k, ya);
                    } else {
#pragma unroll
                        for (int j = 0; j < kBM / 64; ++j)
                            ptx::tma_load_2d(sa + j * kMnBlockBytes, ma, &full[stage], m0 + shp.a_off_mn + 64 * j, ya);
                    }
                    // B's outer coordinate: N (K-major) or K (MN-major)
                    int yb = B_MN ? k0 + shp.b_off_k : n0 + shp.b_off_mn;
                    const CUtensorMap *mb = &tmB;
                    if constexpr (kChunk == kChunkB) {
                        mb = cur.map;
                        yb = cur.y;
                    }
                    if constexpr ((kChunk == kChunkA && A_MN) || (kChunk == kChunkB && B_MN)) cur.advance(cs, kBK);
                    if (!B_MN) {
                        if constexpr (Epi::kGated) {
                            // two boxes of BN/2 rows: the gate rows, then the up rows
                            ptx::tma_load_2d(sb, mb, &full[stage], k0 + shp.b_off_k, yb);
                            ptx::tma_load_2d(sb + (BN / 2) * kRowBytes, mb, &full[stage], k0 + shp.b_off_k,
                                             n0 + shp.b_gate_off + shp.b_off_mn);
                        } else {
                            ptx::tma_load_2d(sb, mb, &full[stage], k0 + shp.b_off_k, yb);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j) {
                            // gated: blocks j >= BN/128 are the up columns
                            const int col = Epi::kGated && j >= BN / 128
                                                ? n0 + shp.b_gate_off + 64 * (j - BN / 128)
                                                : n0 + 64 * j;
                            ptx::tma_load_2d(sb + j * kMnBlockBytes, mb, &full[stage], col + shp.b_off_mn, yb);
                        }
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
                        // K-major: step 32 bytes inside the swizzled row; MN-major:
                        // step kUmmaK whole rows (kUmmaK * 128 bytes)
                        const uint64_t ad = A_MN ? ptx::sdesc_sw128(sa + kk * (kUmmaK * kRowBytes), kMnBlockBytes, 1024)
                                                 : ptx::sdesc_sw128(sa + kk * 32, 16, 1024);
                        const uint64_t bd = B_MN ? ptx::sdesc_sw128(sb + kk * (kUmmaK * kRowBytes), kMnBlockBytes, 1024)
                                                 : ptx::sdesc_sw128(sb + kk * 32, 16, 1024);
                        if constexpr (std::is_same<ElemT, float>::value)
                            ptx::mma_tf32(d_tmem, ad, bd, kIdesc, (kb | kk) != 0 ? 1u : 0u);
                        else
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
        const int ew = warp - 2;                 // epilogue warp index
        const int quarter = warp & 3;            // TMEM lanes this warp may access
        const int group = ew / 4;                // which share of the tile's columns
        const int c0 = group * kChunks / kGroups;
        const int c1 = (group + 1) * kChunks / kGroups;
        EpiWarp w{staging + ew * EpiSmem<Epi>::kWarpBytes, in_bars + 2 * ew, 0, false, 0u, 0u};
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, shp, mb, nb);
            const int row0 = mb * kBM + quarter * 32;  // first output row of this warp
            const int n0 = nb * kTileN;
            epi_issue_input<Epi>(w, ep, &tmIn, lane, n0 + c0 * 32, row0);
            // the decision to go on must be warp-uniform: the TMEM loads are warp-collective
            const bool ok = ptx::mbar_wait(&tfull[acc], acc_phase, abort_flag, err, 4);
            if (!__all_sync(0xffffffffu, ok)) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + acc * BN + (static_cast<uint32_t>(quarter * 32) << 16);
            typename Epi::Row rs;
            if (!epi_tile<Epi, kChunk>(ep, shp, TmemAcc{taddr}, BN / 2, row0, n0, c0, c1, lane, w, rs, true, true,
                                       &tmC0, &tmC1,
                                       &tmIn, &cs, abort_flag, err))
                break;
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1;
        }
        // every output this warp staged has been written, and every input load landed, before the CTA exits
        if (kOuts > 0 && lane == 0) ptx::bulk_wait_all();
        epi_drain_inputs<Epi>(w);
        __syncwarp();
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
