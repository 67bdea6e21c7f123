// runtime.cu -- status codes, the vocabulary padding rule, the device status
// word, kernel timing, TMA tensor-map encoding, SM count, and the column-sum
// kernels for the bias gradients.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "host.h"

namespace tpce {

// ------------------------------------------------------------------ status word
// First device-side failure of any kernel of this library on this device.
__device__ uint32_t g_error_word;

uint32_t *device_error_word() {
    static std::mutex mu;
    static uint32_t *addr[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        addr[dev] = static_cast<uint32_t *>(p);
    }
    return addr[dev];
}

int num_sms() {
    static std::mutex mu;
    static int count[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> g(mu);
    if (!count[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        count[dev] = n;
    }
    return count[dev];
}

// ------------------------------------------------------------------ failure-path test knob
namespace {
std::atomic<int> g_debug_withhold{0};
}

int take_debug_withhold() { return g_debug_withhold.exchange(0); }

// ------------------------------------------------------------------ error text
namespace {
thread_local char g_last_error[512] = "";
}

tpce_status fail(tpce_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

tpce_status fail_cuda(cudaError_t e, const char *what) {
    return fail(TPCE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool sync_check_enabled() {
    static int on = -1;
    if (on < 0) {
        const char *v = getenv("TPCE_SYNC_CHECK");
        on = (v && v[0] == '1') ? 1 : 0;
    }
    return on == 1;
}

tpce_status check_launch(const char *name, cudaStream_t s) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail_cuda(e, name);
    if (sync_check_enabled()) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if ((e = cudaStreamIsCapturing(s, &cs)) != cudaSuccess) return fail_cuda(e, name);
        if (cs == cudaStreamCaptureStatusNone && (e = cudaDeviceSynchronize()) != cudaSuccess) return fail_cuda(e, name);
    }
    return TPCE_OK;
}

// ------------------------------------------------------------------ tensor maps
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool make_tmap(CUtensorMap *m, int dt, const void *base, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer, int swizzle) {
    auto fn = encode_fn();
    const uint64_t esz = dt == 1 ? 4 : 2;
    if (!fn || inner == 0 || outer == 0 || !aligned16(base) || (ld * esz) % 16 != 0) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {ld * esz};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, dt == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ profiling
namespace {
struct Rec {
    const char *name;
    int dev;
    cudaEvent_t a, b;
};
struct Agg {
    const char *name;
    int64_t launches;
    double ms;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<Rec> g_recs;
std::vector<Agg> g_agg;
std::map<int, std::vector<cudaEvent_t>> g_pool;

cudaEvent_t take_event(int dev) {
    auto &v = g_pool[dev];
    if (!v.empty()) {
        cudaEvent_t e = v.back();
        v.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    return e;
}

void release_records() {
    for (auto &r : g_recs) {
        if (r.a) g_pool[r.dev].push_back(r.a);
        if (r.b) g_pool[r.dev].push_back(r.b);
    }
    g_recs.clear();
}
}  // namespace

KernelTimer::KernelTimer(const char *name, cudaStream_t stream) : name_(name), stream_(stream) {
    if (!name_) return;  // an untimed launch
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (!g_prof_on) return;
    int dev = 0;
    cudaGetDevice(&dev);
    start_ = take_event(dev);
    if (start_ && cudaEventRecord(start_, stream_) != cudaSuccess) {
        g_pool[dev].push_back(start_);
        start_ = nullptr;
    }
}

KernelTimer::~KernelTimer() {
    if (!start_) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    int dev = 0;
    cudaGetDevice(&dev);
    cudaEvent_t end = take_event(dev);
    if (!end || cudaEventRecord(end, stream_) != cudaSuccess) {
        g_pool[dev].push_back(start_);
        if (end) g_pool[dev].push_back(end);
        return;
    }
    g_recs.push_back({name_, dev, start_, end});
}

// ------------------------------------------------------------------ column sums
__device__ __forceinline__ void add8(const __nv_bfloat16 *p, float *acc) {
    uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 f = __bfloat1622float2(h[i]);
        acc[2 * i] += f.x;
        acc[2 * i + 1] += f.y;
    }
}
__device__ __forceinline__ void add8(const float *p, float *acc) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
}

// Row addressing of the column sum's input: one [R, N] matrix with row pitch
// ld, or its rows split over sequence-chunk buffers of `rows` rows each.
template <typename T>
struct DenseRows {
    const T *X;
    int64_t ld;
    __device__ const T *row(int64_t r) const { return X + r * ld; }
};
template <typename T>
struct ChunkedRows {
    const T *p[kMaxRowChunks];
    int64_t rows, ld;
    __device__ const T *row(int64_t r) const {
        const int64_t c = r / rows;
        return p[c] + (r - c * rows) * ld;
    }
};

// Stage 1: block (x, y) sums rows [y*rows_per, (y+1)*rows_per) of 256 columns
// starting at 256*x; each lane owns 8 adjacent columns (one vector load per
// row), the 8 warps stride over the rows four rows at a time (four loads in
// flight per lane: the pass is HBM-bound), and shared memory combines the
// warps.
template <typename T, class Rows>
__global__ void __launch_bounds__(256) colsum_stage1(const Rows rows_of, int64_t R, int64_t N, int64_t rows_per,
                                                     float *__restrict__ part) {
    __shared__ float red[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 256 + lane * 8;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * rows_per;
    const int64_t r1 = min(R, r0 + rows_per);
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    if (c0 < N) {
        int64_t r = r0 + warp;
        for (; r + 24 < r1; r += 32) {
            float a0[8] = {0, 0, 0, 0, 0, 0, 0, 0}, a1[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            float a2[8] = {0, 0, 0, 0, 0, 0, 0, 0}, a3[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            add8(rows_of.row(r) + c0, a0);
            add8(rows_of.row(r + 8) + c0, a1);
            add8(rows_of.row(r + 16) + c0, a2);
            add8(rows_of.row(r + 24) + c0, a3);
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] += (a0[i] + a1[i]) + (a2[i] + a3[i]);
        }
        for (; r < r1; r += 8) add8(rows_of.row(r) + c0, acc);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) red[warp][lane * 8 + i] = acc[i];
    __syncthreads();
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;
    if (c < N) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][threadIdx.x];
        part[static_cast<int64_t>(blockIdx.y) * N + c] = s;
    }
}

// Stage 2: out[c] = sum over the S partial rows.
__global__ void colsum_stage2(const float *__restrict__ part, int S, int64_t N, float *__restrict__ out) {
    const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= N) return;
    float s = 0.0f;
    for (int i = 0; i < S; ++i) s += part[static_cast<int64_t>(i) * N + c];
    out[c] = s;
}

// Row splits of the column sum: enough blocks to cover the SMs about four times
// (with four row loads in flight per lane, enough bytes in flight to fill HBM).
// Fixed (not queried from the device) so workspace sizes are known on the host.
constexpr int64_t kColsumTargetBlocks = 4 * 152;

static int colsum_splits(int64_t R, int64_t N) {
    const int64_t col_blocks = (N + 255) / 256;
    int64_t S = (kColsumTargetBlocks + col_blocks - 1) / col_blocks;
    S = std::max<int64_t>(1, std::min<int64_t>(S, 64));
    S = std::min<int64_t>(S, std::max<int64_t>(1, R));
    return static_cast<int>(S);
}

size_t colsum_partial_floats(int64_t R, int64_t N) { return static_cast<size_t>(colsum_splits(R, N)) * N; }

template <class Rows>
static tpce_status colsum_impl(const Rows &rows_of, int64_t R, int64_t N, float *out, float *partial, cudaStream_t s) {
    if (N <= 0) return TPCE_OK;
    if (R <= 0) return cuda_status(cudaMemsetAsync(out, 0, sizeof(float) * N, s));
    const int S = colsum_splits(R, N);
    const int64_t rows_per = (R + S - 1) / S;
    {
        KernelTimer t("colsum_stage1", s);
        dim3 grid(static_cast<unsigned>((N + 255) / 256), static_cast<unsigned>(S));
        using T = typename std::remove_const<typename std::remove_pointer<decltype(rows_of.row(0))>::type>::type;
        colsum_stage1<T, Rows><<<grid, 256, 0, s>>>(rows_of, R, N, rows_per, partial);
        if (check_launch("colsum_stage1", s) != TPCE_OK) return TPCE_ERR_CUDA;
    }
    {
        KernelTimer t("colsum_stage2", s);
        colsum_stage2<<<static_cast<unsigned>((N + 255) / 256), 256, 0, s>>>(partial, S, N, out);
        if (check_launch("colsum_stage2", s) != TPCE_OK) return TPCE_ERR_CUDA;
    }
    return TPCE_OK;
}

tpce_status colsum(int dt, const void *X, int64_t R, int64_t N, int64_t ld, float *out, float *partial,
                   cudaStream_t s) {
    if (dt == 1) return colsum_impl(DenseRows<float>{static_cast<const float *>(X), ld}, R, N, out, partial, s);
    return colsum_impl(DenseRows<__nv_bfloat16>{static_cast<const __nv_bfloat16 *>(X), ld}, R, N, out, partial, s);
}

tpce_status colsum_chunks(int dt, const void *const *chunks, int count, int64_t rows, int64_t N, int64_t ld,
                          float *out, float *partial, cudaStream_t s) {
    if (count < 1 || count > kMaxRowChunks || rows < 1) return TPCE_ERR_INVALID;
    if (dt == 1) {
        ChunkedRows<float> c{};
        for (int i = 0; i < count; ++i) c.p[i] = static_cast<const float *>(chunks[i]);
        c.rows = rows;
        c.ld = ld;
        return colsum_impl(c, rows * count, N, out, partial, s);
    }
    ChunkedRows<__nv_bfloat16> c{};
    for (int i = 0; i < count; ++i) c.p[i] = static_cast<const __nv_bfloat16 *>(chunks[i]);
    c.rows = rows;
    c.ld = ld;
    return colsum_impl(c, rows * count, N, out, partial, s);
}

// ------------------------------------------------------------------ fp32 -> bf16
__global__ void f32_to_bf16_kernel(const float4 *__restrict__ in, uint4 *__restrict__ out, int64_t n8) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = __ldg(in + 2 * i), b = __ldg(in + 2 * i + 1);
        __nv_bfloat162 h0 = __floats2bfloat162_rn(a.x, a.y), h1 = __floats2bfloat162_rn(a.z, a.w);
        __nv_bfloat162 h2 = __floats2bfloat162_rn(b.x, b.y), h3 = __floats2bfloat162_rn(b.z, b.w);
        uint4 u;
        u.x = *reinterpret_cast<uint32_t *>(&h0);
        u.y = *reinterpret_cast<uint32_t *>(&h1);
        u.z = *reinterpret_cast<uint32_t *>(&h2);
        u.w = *reinterpret_cast<uint32_t *>(&h3);
        out[i] = u;
    }
}

tpce_status f32_to_bf16(const float *in, void *out, int64_t n, cudaStream_t s) {
    if (n <= 0) return TPCE_OK;
    const int64_t n8 = n / 8;
    const int sms = num_sms();
    const int64_t blocks = std::min<int64_t>((n8 + 255) / 256, static_cast<int64_t>(std::max(sms, 1)) * 8);
    KernelTimer t("f32_to_bf16", s);
    f32_to_bf16_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(reinterpret_cast<const float4 *>(in),
                                                                     static_cast<uint4 *>(out), n8);
    return check_launch("f32_to_bf16", s);
}

// ------------------------------------------------------------------ transpose
// 32 x 32 tiles through shared memory (one padding column avoids bank conflicts).
__global__ void __launch_bounds__(256) transpose_f32_kernel(const float *__restrict__ in, int64_t R, int64_t C,
                                                            int64_t ld_in, float *__restrict__ out, int64_t ld_out) {
    __shared__ float tile[32][33];
    const int64_t c = static_cast<int64_t>(blockIdx.x) * 32 + threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32;
    for (int j = threadIdx.y; j < 32; j += 8) {
        const int64_t r = r0 + j;
        if (r < R && c < C) tile[j][threadIdx.x] = in[r * ld_in + c];
    }
    __syncthreads();
    const int64_t orow = static_cast<int64_t>(blockIdx.x) * 32;  // output row = input column
    const int64_t ocol = r0 + threadIdx.x;                       // output column = input row
    for (int j = threadIdx.y; j < 32; j += 8) {
        if (orow + j < C && ocol < R) out[(orow + j) * ld_out + ocol] = tile[threadIdx.x][j];
    }
}

// bf16 transpose out[c, r] = in[r, c] through 64 x 64 tiles in shared memory,
// 16-byte loads and stores on both sides so that every global access is a
// whole 128-byte row of the tile. In shared memory the 16-byte pieces of tile
// row r are permuted by (r >> 3) & 7, so that the 8 threads that gather one
// 16-byte output piece from 8 tile rows j*8 + e (one per j) read 8 different
// bank groups. Input rows r >= R read as zeros; each output row is written up
// to column out_cols = R rounded up to 8, so that padding holds zeros.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint4 *__restrict__ in, int64_t R, int64_t C,
                                                             int64_t ld_in8, uint4 *__restrict__ out, int64_t out_cols,
                                                             int64_t ld_out8) {
    __shared__ __align__(16) uint8_t tile[64 * 128];
    const int t = threadIdx.x;
    const int64_t r0 = static_cast<int64_t>(blockIdx.y) * 64;
    const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int row = p * 32 + (t >> 3), ch = t & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (r0 + row < R && c0 + ch * 8 < C) v = __ldg(in + (r0 + row) * ld_in8 + (c0 >> 3) + ch);
        *reinterpret_cast<uint4 *>(tile + row * 128 + ((ch ^ ((row >> 3) & 7)) << 4)) = v;
    }
    __syncthreads();
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int oc = p * 32 + (t >> 3), j = t & 7;  // output row c0 + oc, its 16-byte piece j
        if (c0 + oc >= C || r0 + j * 8 >= out_cols) continue;
        uint16_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int row = j * 8 + e;  // (row >> 3) & 7 == j
            h[e] = *reinterpret_cast<const uint16_t *>(tile + row * 128 + ((((oc >> 3) ^ j)) << 4) + ((oc & 7) << 1));
        }
        uint4 v;
        v.x = h[0] | (static_cast<uint32_t>(h[1]) << 16);
        v.y = h[2] | (static_cast<uint32_t>(h[3]) << 16);
        v.z = h[4] | (static_cast<uint32_t>(h[5]) << 16);
        v.w = h[6] | (static_cast<uint32_t>(h[7]) << 16);
        out[(c0 + oc) * ld_out8 + (r0 >> 3) + j] = v;
    }
}

tpce_status transpose_bf16(const void *in, int64_t R, int64_t C, int64_t ld_in, void *out, int64_t ld_out,
                           cudaStream_t s) {
    if (R <= 0 || C <= 0) return TPCE_OK;
    const int64_t out_cols = (R + 7) / 8 * 8;
    if (C % 8 || ld_in % 8 || ld_out % 8 || ld_out < out_cols || !aligned16(in) || !aligned16(out))
        return fail(TPCE_ERR_INVALID, "transpose_bf16: rows of 8-element multiples, 16-byte aligned");
    KernelTimer t("transpose_bf16", s);
    dim3 grid(static_cast<unsigned>((C + 63) / 64), static_cast<unsigned>((R + 63) / 64));
    if (grid.y > 65535) return fail(TPCE_ERR_SHAPE, "transpose_bf16: %lld rows", static_cast<long long>(R));
    transpose_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4 *>(in), R, C, ld_in / 8,
                                               static_cast<uint4 *>(out), out_cols, ld_out / 8);
    return check_launch("transpose_bf16", s);
}

tpce_status transpose_f32(const float *in, int64_t R, int64_t C, int64_t ld_in, float *out, int64_t ld_out,
                          cudaStream_t s) {
    if (R <= 0 || C <= 0) return TPCE_OK;
    KernelTimer t("transpose_f32", s);
    dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((R + 31) / 32));
    transpose_f32_kernel<<<grid, dim3(32, 8), 0, s>>>(in, R, C, ld_in, out, ld_out);
    return check_launch("transpose_f32", s);
}

}  // namespace tpce

// ====================================================================== C ABI
using namespace tpce;

extern "C" const char *tpce_status_string(tpce_status s) {
    switch (s) {
        case TPCE_OK: return "TPCE_OK";
        case TPCE_ERR_INVALID: return "TPCE_ERR_INVALID";
        case TPCE_ERR_SHAPE: return "TPCE_ERR_SHAPE";
        case TPCE_ERR_ALIGN: return "TPCE_ERR_ALIGN";
        case TPCE_ERR_WORKSPACE: return "TPCE_ERR_WORKSPACE";
        case TPCE_ERR_CUDA: return "TPCE_ERR_CUDA";
        case TPCE_ERR_TIMEOUT: return "TPCE_ERR_TIMEOUT";
        case TPCE_ERR_UNSUPPORTED: return "TPCE_ERR_UNSUPPORTED";
    }
    return "TPCE_ERR_UNKNOWN";
}

extern "C" int tpce_version(void) { return 100; }

extern "C" const char *tpce_last_error(void) { return g_last_error; }

extern "C" int64_t tpce_pad_vocab(int64_t v, int t, int divisor) {
    if (v < 0 || t < 1 || divisor < 1) return -1;
    const int64_t m = static_cast<int64_t>(divisor) * t;
    return (v + m - 1) / m * m;
}

extern "C" tpce_status tpce_device_status(void *stream, int clear, uint32_t *detail) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return TPCE_ERR_CUDA;
    uint32_t *w = device_error_word();
    if (!w) return TPCE_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, w, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TPCE_ERR_CUDA;
    if (clear && cudaMemset(w, 0, sizeof(uint32_t)) != cudaSuccess) return TPCE_ERR_CUDA;
    if (detail) *detail = v;
    const uint32_t code = v & 0xffu;
    return code <= TPCE_ERR_UNSUPPORTED ? static_cast<tpce_status>(code) : TPCE_ERR_INVALID;
}

extern "C" tpce_status tpce_debug_withhold_next_load(int on) {
    g_debug_withhold.store(on ? 1 : 0);
    return TPCE_OK;
}

extern "C" tpce_status tpce_profile_enable(int on) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    release_records();
    g_agg.clear();
    g_prof_on = on != 0;
    return TPCE_OK;
}

extern "C" int tpce_profile_count(void) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    std::vector<Agg> agg;
    int bad = 0;
    for (auto &r : g_recs) {
        float ms = 0.0f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) {
            ++bad;
            continue;
        }
        auto it = std::find_if(agg.begin(), agg.end(),
                               [&](const Agg &x) { return std::string(x.name) == std::string(r.name); });
        if (it == agg.end())
            agg.push_back({r.name, 1, ms});
        else {
            it->launches += 1;
            it->ms += ms;
        }
    }
    release_records();
    // keep aggregating across calls until the next tpce_profile_enable
    for (auto &a : agg) {
        auto it = std::find_if(g_agg.begin(), g_agg.end(),
                               [&](const Agg &x) { return std::string(x.name) == std::string(a.name); });
        if (it == g_agg.end())
            g_agg.push_back(a);
        else {
            it->launches += a.launches;
            it->ms += a.ms;
        }
    }
    return bad ? -1 : static_cast<int>(g_agg.size());
}

extern "C" tpce_status tpce_profile_get(int i, const char **name, int64_t *launches, double *total_ms) {
    std::lock_guard<std::mutex> g(g_prof_mu);
    if (i < 0 || i >= static_cast<int>(g_agg.size())) return TPCE_ERR_INVALID;
    if (name) *name = g_agg[i].name;
    if (launches) *launches = g_agg[i].launches;
    if (total_ms) *total_ms = g_agg[i].ms;
    return TPCE_OK;
}

extern "C" size_t tpce_tail_workspace_bytes(void) { return tpce::kTailScratchBytes; }
