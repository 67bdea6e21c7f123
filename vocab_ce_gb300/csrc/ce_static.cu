// ce_static.cu -- vocab_parallel_ce_loss_static: the forward of the fused
// vocabulary-parallel cross-entropy (loss and lse, no gradients) with its
// scratch in a static device array instead of a caller-provided workspace.
//
// Who needs it: a caller that cannot call cudaMalloc -- for instance a plugin
// running inside a host framework whose memory planner owns every device
// buffer and forbids allocations it did not plan, or a latency-critical path
// that must not risk the implicit device synchronisation a cudaMalloc may
// perform. Such a caller still passes its inputs and outputs; everything
// else the call needs lives in the static array below.
//
// The scratch is a file-scope __device__ array of TPCE_CE_STATIC_SCRATCH_BYTES
// bytes: every GPU that loads this library holds it until the process exits.
// Host code cannot use the array's name as a device address (on the host it
// names a host-side stand-in), so the first call on each device, with that
// device current, asks the runtime for the array's device address with
// cudaGetSymbolAddress and caches it. Under CUDA's default lazy module
// loading that lookup is also where this file's module -- and with it the
// array's memory -- is loaded onto the device (under eager loading it happens
// when the library's modules load), so the first call per device commits the
// array once, an implicit device allocation that can fail when the device is
// already full. Make that first call before a memory planner reserves the
// device, and before any stream capture; later calls allocate nothing. All
// calls share the one array: two calls whose kernels overlap on the GPU
// (different streams, no ordering) race on it. The array keeps the last
// call's contents. Every statistic the combine kernel reads is written earlier
// in the same call; the one thing that must start at zero, the tickets of the
// fold of a shard's partial statistics, is cleared by each call (a memset on
// its stream) before its logit GEMM. The statistics are vocab_parallel_ce's:
// one (max, sumexp) pair per shard and token, reached through a few partial
// pairs per shard where the shard is cut into parts, so the 129K-vocabulary
// config (16,384 tokens, t = 8, 9 parts per shard) needs 10.6 MB of the array.
#include <cuda_runtime.h>

#include <mutex>

#include "ce_common.cuh"
#include "gemm_launch.cuh"
#include "host.h"

namespace tpce {

static __device__ __align__(256) unsigned char g_ce_static_scratch[TPCE_CE_STATIC_SCRATCH_BYTES];

namespace {

// The array's device address on the current device, looked up once per device.
tpce_status static_scratch_address(uint8_t **out) {
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "vocab_parallel_ce_loss_static: cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(TPCE_ERR_CUDA, "vocab_parallel_ce_loss_static: device %d out of range", dev);
    std::lock_guard<std::mutex> g(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_ce_static_scratch);
        if (e != cudaSuccess) return fail_cuda(e, "vocab_parallel_ce_loss_static: cudaGetSymbolAddress");
        addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(addr[dev]);
    return TPCE_OK;
}

}  // namespace
}  // namespace tpce

using namespace tpce;

extern "C" tpce_status vocab_parallel_ce_loss_static(const void *H, const void *E, const int32_t *targets, int64_t T,
                                                     int64_t h, int64_t v_pad, int64_t v_valid, int t, int dtype,
                                                     float *loss, float *lse, void *stream) {
    tpce_status st = check_ce_shape(T, h, v_pad, v_valid, t, dtype);
    if (st != TPCE_OK) return st;
    if (T == 0) return TPCE_OK;
    if (!H || !E || !targets || !loss) return TPCE_ERR_INVALID;
    if (!aligned16(H) || !aligned16(E)) return TPCE_ERR_ALIGN;
    for (const void *p : {static_cast<const void *>(targets), static_cast<const void *>(loss),
                          static_cast<const void *>(lse)})
        if (reinterpret_cast<uintptr_t>(p) & 3u) return TPCE_ERR_ALIGN;

    // scratch layout (vocab_parallel_ce's): the shards' (max, sumexp) [t][T],
    // the parts' pairs and tickets when shards are cut into parts, target
    // logit [T], lse [T] if not an output
    const bool f32 = dtype == TPCE_F32;
    const CeStatsPlan P = ce_stats_plan(T, v_pad, t, dtype, TPCE_PAIR_BN == 256);
    const size_t stats_bytes = round_up(static_cast<size_t>(t) * T * sizeof(float2), 256);
    const size_t parts_bytes = round_up(ce_parts_bytes(P, T), 256);
    const size_t ticket_bytes = ce_ticket_bytes(P, T, t);
    const size_t tau_bytes = round_up(static_cast<size_t>(T) * sizeof(float), 256);
    const size_t lse_bytes = lse ? 0 : tau_bytes;
    const size_t need = stats_bytes + parts_bytes + round_up(ticket_bytes, 256) + tau_bytes + lse_bytes;
    if (need > TPCE_CE_STATIC_SCRATCH_BYTES)
        return fail(TPCE_ERR_WORKSPACE,
                    "vocab_parallel_ce_loss_static: T=%lld and %lld statistics parts per token need %zu bytes of "
                    "scratch; the static scratch holds %u",
                    static_cast<long long>(T), static_cast<long long>(P.parts), need,
                    static_cast<unsigned>(TPCE_CE_STATIC_SCRATCH_BYTES));
    uint8_t *base = nullptr;
    st = static_scratch_address(&base);
    if (st != TPCE_OK) return st;
    float2 *stats = reinterpret_cast<float2 *>(base);
    float2 *parts = reinterpret_cast<float2 *>(base + stats_bytes);
    uint32_t *tickets = reinterpret_cast<uint32_t *>(base + stats_bytes + parts_bytes);
    uint8_t *rest = base + stats_bytes + parts_bytes + round_up(ticket_bytes, 256);
    float *tau = reinterpret_cast<float *>(rest);
    float *lse_buf = lse ? lse : reinterpret_cast<float *>(rest + tau_bytes);
    uint32_t *err = device_error_word();
    if (!err) return fail(TPCE_ERR_CUDA, "vocab_parallel_ce_loss_static: device status word");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int Ti = static_cast<int>(T), hi = static_cast<int>(h), vpi = static_cast<int>(v_pad);
    const int vvi = static_cast<int>(v_valid);

    Operand a{H, T, h, h};      // K-major [T, h]
    Operand b{E, v_pad, h, h};  // K-major: N = v_pad rows, K = h columns
    // the tickets keep the last call's contents: clear them (a memset, not an allocation)
    if (ticket_bytes && cudaMemsetAsync(tickets, 0, ticket_bytes, s) != cudaSuccess)
        return fail(TPCE_ERR_CUDA, "vocab_parallel_ce_loss_static: cudaMemsetAsync of the statistics tickets");
    EpiCeStats::Params ep{stats, parts, tickets, tau, targets, T, vvi, 0, 0, P.bn, P.run_len, P.parts_per_shard, t};
    if (f32)
        st = launch_gemm<float, 128, false, false, EpiCeStats>("ce_static_logits_stats", a, b, nullptr, nullptr, Ti, vpi, hi, 0, 0, 0,
                                                               0, ep, s, /*timed=*/false);
    else if (P.pair)  // no tail scratch: the CTA pairs never split a tile here
        st = launch_gemm_pair<256, false, false, EpiCeStats>("ce_static_logits_stats", a, b, nullptr, nullptr, Ti, vpi, hi,
                                                             0, 0, 0, 0, ep, s, /*timed=*/false, 0, nullptr, nullptr,
                                                             P.run_len);
    else if (P.bn == 256)
        st = launch_gemm<__nv_bfloat16, 256, false, false, EpiCeStats>("ce_static_logits_stats", a, b, nullptr, nullptr, Ti,
                                                                       vpi, hi, 0, 0, 0, 0, ep, s, /*timed=*/false);
    else
        st = launch_gemm<__nv_bfloat16, 128, false, false, EpiCeStats>("ce_static_logits_stats", a, b, nullptr, nullptr, Ti, vpi, hi,
                                                                       0, 0, 0, 0, ep, s, /*timed=*/false);
    if (st != TPCE_OK) return st;
    launch_ce_combine(stats, tau, targets, T, t, 1, vvi, loss, lse_buf, err, s);
    return check_launch("ce_static_combine", s);
}
