// host.h -- host-side pieces shared by the translation units of libtpce:
// device status word, SM count, kernel timing, TMA tensor maps, validation
// helpers and the column-sum kernels used for the bias gradients.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "tpce.h"

namespace tpce {

// address of the device status word on the current device (null on failure)
uint32_t *device_error_word();
// number of SMs of the current device (0 on failure)
int num_sms();
// 1 once after tpce_debug_withhold_next_load(1) armed it (the arming is used
// up by the CTA-pair GEMM launch that reads it), else 0.
int take_debug_withhold();

// RAII kernel timer: when profiling is on, records an event pair around the
// launches made during its lifetime on `stream` and files them under `name`.
// A null name makes it inert.
class KernelTimer {
   public:
    KernelTimer(const char *name, cudaStream_t stream);
    ~KernelTimer();
    KernelTimer(const KernelTimer &) = delete;
    KernelTimer &operator=(const KernelTimer &) = delete;

   private:
    const char *name_;
    cudaStream_t stream_;
    cudaEvent_t start_ = nullptr;
};

// 2-D tensor map over bf16 (dt 0) or fp32 (dt 1) data: `inner` contiguous
// elements per row (row pitch `ld` elements), `outer` rows, box
// {box_inner, box_outer}, shared-memory swizzle of 128 or 64 bytes.
bool make_tmap(CUtensorMap *m, int dt, const void *base, uint64_t inner, uint64_t outer, uint64_t ld,
               uint32_t box_inner, uint32_t box_outer, int swizzle = 128);

// fp32 -> bf16, n elements (n % 8 == 0, 16-byte aligned)
tpce_status f32_to_bf16(const float *in, void *out, int64_t n, cudaStream_t s);

// fp32 column sums out[n] = sum_r X[r, n] of a bf16 (dt 0) or fp32 (dt 1)
// [R, N] matrix (row pitch ld), through a partial buffer of
// colsum_partial_floats(R, N) floats.
size_t colsum_partial_floats(int64_t R, int64_t N);
tpce_status colsum(int dt, const void *X, int64_t R, int64_t N, int64_t ld, float *out, float *partial,
                   cudaStream_t s);
// Workspace the GEMMs use to split the last partial wave of tiles along K:
// at most kTailMaxUnits parts of one CTA pair's 256 x 256 fp32 tile, plus
// their tickets. Every workspace layout starts with this region.
constexpr int kTailMaxUnits = 64;
constexpr size_t kTailScratchBytes = static_cast<size_t>(kTailMaxUnits) * 2 * 128 * 256 * 4 + 4096;

// The same over rows split into `count` buffers of `rows` rows each (row
// pitch ld): the column sums of their concatenation. count <= kMaxRowChunks.
constexpr int kMaxRowChunks = 16;
tpce_status colsum_chunks(int dt, const void *const *chunks, int count, int64_t rows, int64_t N, int64_t ld,
                          float *out, float *partial, cudaStream_t s);

// out[c, r] = in[r, c] for a bf16 [R, C] matrix (row pitches ld_in, ld_out,
// in elements): C, ld_in and ld_out multiples of 8, 16-byte aligned pointers,
// ld_out >= R8 = R rounded up to 8. Output columns R .. R8 are written as
// zeros; columns from R8 on are not touched (so an output block may sit inside
// a wider matrix).
tpce_status transpose_bf16(const void *in, int64_t R, int64_t C, int64_t ld_in, void *out, int64_t ld_out,
                           cudaStream_t s);
// out[c, r] = in[r, c] for an fp32 [R, C] matrix (row pitches ld_in, ld_out).
tpce_status transpose_f32(const float *in, int64_t R, int64_t C, int64_t ld_in, float *out, int64_t ld_out,
                          cudaStream_t s);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline tpce_status cuda_status(cudaError_t e) { return e == cudaSuccess ? TPCE_OK : TPCE_ERR_CUDA; }

// Record a description of a failure for tpce_last_error() (per host thread)
// and return `st`.
tpce_status fail(tpce_status st, const char *fmt, ...);
tpce_status fail_cuda(cudaError_t e, const char *what);
// cudaGetLastError after a launch on stream s, recorded under the kernel's name
tpce_status check_launch(const char *name, cudaStream_t s);
// when the environment sets TPCE_SYNC_CHECK=1, every launch is followed by a
// device synchronisation so that a failing kernel is named by check_launch --
// except while s is being captured into a CUDA graph, where synchronising is
// not allowed
bool sync_check_enabled();

}  // namespace tpce
