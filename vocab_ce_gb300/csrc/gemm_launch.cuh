// gemm_launch.cuh -- host-side launch of tc_gemm_kernel: tensor maps, tile
// width, rasterisation and the persistent grid size.
#pragma once

#include <algorithm>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "gemm.cuh"
#include "gemm_pair.cuh"
#include "host.h"

namespace tpce {
namespace {

// An operand as it sits in memory (row-major, row pitch `ld` elements).
// K-major operand: `rows` = extent of the output dimension it feeds (M for A,
// N for B), `cols` = contraction extent. MN-major operand: `rows` =
// contraction extent, `cols` = output-dimension extent.
struct Operand {
    const void *ptr;
    int64_t rows, cols, ld;
};

// An output the epilogue writes with TMA stores: [rows, cols], row pitch ld
// elements of the epilogue's output type.
struct OutView {
    void *ptr;
    int64_t rows, cols, ld;
};

// The rows of the chunked role of a launch (see ChunkSet) in separate
// buffers: `count` device pointers (a host array, read during the launch
// only), each holding `rows` rows with the role's row pitch and columns.
struct Chunks {
    const void *const *ptrs;
    int64_t rows;
    int count;
};

// Scratch for the split tail of a CTA-pair launch (caller's workspace);
// null or too small: the tail is not split.
struct TailScratch {
    void *ptr;
    size_t bytes;
};

// Split-tail plan. With C clusters and tiles = W C + r, the last r tiles (a
// partial wave, r <= C / 2) are each split along K into s parts, so the last
// wave runs r s parts of 1/s the work on otherwise idle clusters. s is capped
// so that every part has at least kTailMinKBlocks K blocks, r s <= C (one
// part per cluster) and r s <= kTailMaxUnits (the scratch bound).
// Measured on GB300 (A/B, two repetitions): 32 K blocks per part is best --
// the 8.3B step's dH GEMM gains 10% and its GEMM2 / dX 7%, while splitting
// the K = 3072 GEMMs (16-block parts) did not pay for the partials' round
// trip through L2.
#ifndef TPCE_TAIL_MIN_KBLOCKS
#define TPCE_TAIL_MIN_KBLOCKS 32
#endif
#ifndef TPCE_TAIL_SPLIT
#define TPCE_TAIL_SPLIT 1
#endif
constexpr int kTailMinKBlocks = TPCE_TAIL_MIN_KBLOCKS;  // build-time tuning knobs
constexpr int kTailMaxSplit = 8;
inline void plan_tail(GemmShape &s, int clusters, int bn, const TailScratch *ts, cudaStream_t stream, bool &memset_ok) {
    const int tiles = s.tiles_m * s.unit_cols;  // work units: tiles, or runs of tiles
    s.full_units = tiles;
    s.split = 1;
    s.tail_tiles = 0;
    s.partial = nullptr;
    s.tickets = nullptr;
    memset_ok = true;
    if (!TPCE_TAIL_SPLIT || s.run_len != 1 || !ts || !ts->ptr || clusters < 2 || tiles <= clusters) return;
    const int r = tiles % clusters;
    if (r == 0 || r > clusters / 2) return;
    int sp = std::min({kTailMaxSplit, clusters / r, kTailMaxUnits / r, s.k_blocks / kTailMinKBlocks});
    if (sp < 2) return;
    const size_t part_bytes = sizeof(float) * 2 * kBM * static_cast<size_t>(bn);
    const size_t need = part_bytes * r * sp + sizeof(uint32_t) * 2 * r;
    if (ts->bytes < need) return;
    s.full_units = tiles - r;
    s.split = sp;
    s.tail_tiles = r;
    s.partial = static_cast<float *>(ts->ptr);
    s.tickets = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ts->ptr) + part_bytes * r * sp);
    memset_ok = cudaMemsetAsync(s.tickets, 0, sizeof(uint32_t) * 2 * r, stream) == cudaSuccess;
}

// Tensor maps of the chunks of one role, built like the role's own map.
template <int kChunk, typename Build>
inline bool build_chunk_maps(ChunkSet<kChunk> &cs, const Chunks *ch, Build build) {
    std::memset(static_cast<void *>(&cs), 0, sizeof(cs));
    if constexpr (kChunk == kChunkNone) {
        return ch == nullptr;
    } else {
        if (!ch || ch->count < 1 || ch->count > kMaxChunks || ch->rows <= 0 || ch->rows % 128 != 0 ||
            ch->rows > (1 << 30))
            return false;
        cs.rows = static_cast<int>(ch->rows);
        cs.count = ch->count;
        for (int c = 0; c < ch->count; ++c)
            if (!ch->ptrs[c] || !build(&cs.m[c], ch->ptrs[c], ch->rows)) return false;
        return true;
    }
}

// Tiles are walked in groups of `group_m` row-blocks, row-block fastest, so
// the CTAs of one wave share a few A and B panels in L2. A group's A panels
// (group_m row-blocks x K) are reused by every column block the group walks;
// a panel budget can cap the group so that they stay in L2. Build-time tuning
// knobs: the budget and the smallest group. Default: 16 row-blocks whatever
// K is. Measured on GB300: at K = 8192 the 16-block group re-reads A from
// DRAM (92 GB per 129K-vocabulary logit GEMM against 8.7 GB ideal), yet
// budgets of 16-32 MB with groups of 2-8 were no faster on any workload
// (within +-1.5%, slower on that logit GEMM): the kernels are bound by the
// tensor pipe and the power cap, not by DRAM.
#ifndef TPCE_GROUP_PANEL_BYTES
#define TPCE_GROUP_PANEL_BYTES (64ll << 20)
#endif
#ifndef TPCE_GROUP_MIN
#define TPCE_GROUP_MIN 16
#endif
inline int pick_group_m(int tiles_m, int64_t rows_per_block, int64_t K, int64_t elem_bytes) {
    const int64_t panel = std::max<int64_t>(1, rows_per_block * K * elem_bytes);  // one row-block's A panel
    const int64_t g = std::max<int64_t>(TPCE_GROUP_MIN, std::min<int64_t>(16, TPCE_GROUP_PANEL_BYTES / panel));
    return static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles_m, g)));
}

// L2 eviction priorities of a CTA-pair launch. The group's A panels (group_m
// row-blocks x K) are read once per column block the group walks; B's panels
// once per group. With TPCE_L2_HINT=1, when the A panels fit the budget and B
// is too large to stay in L2 anyway, A's lines are loaded evict_last and B's
// evict_first. Off by default: measured on GB300 (the 70B MLP + 129K CE step,
// A/B twice in one session) it was 2% slower, and the 129K logit-statistics
// GEMM read 77 GB from DRAM instead of 64 GB -- the kept A panels crowd out B
// lines that the other row-blocks of the same wave were still to read.
#ifndef TPCE_L2_HINT
#define TPCE_L2_HINT 0
#endif
#ifndef TPCE_L2_KEEP_BYTES
#define TPCE_L2_KEEP_BYTES (64ll << 20)
#endif
inline int pick_l2_hint(int group_m, int tiles_n, int64_t rows_per_block, int64_t bn, int64_t K, int64_t elem_bytes) {
    const int64_t a_group = group_m * rows_per_block * K * elem_bytes;
    const int64_t b_all = tiles_n * bn * K * elem_bytes;
    return (TPCE_L2_HINT && tiles_n > 1 && a_group <= TPCE_L2_KEEP_BYTES && b_all > TPCE_L2_KEEP_BYTES) ? 1 : 0;
}

// Tile widths a launch may use.
enum : unsigned { kBN128 = 1u, kBN192 = 2u, kBN256 = 4u };
// Build-time tuning knob: the tile widths launch_gemm_auto may choose from.
#ifndef TPCE_BN_MASK
#define TPCE_BN_MASK 7u
#endif

// The tile width that finishes an M x N output soonest: the waves of
// 128 x BN tiles over the SMs times the tile time, taken as BN plus a fixed
// per-tile cost worth 96 columns (fitted on GB300: 192-wide tiles win only
// where they save a whole wave, e.g. N = 3072 on 64 row-blocks, and lose on
// N = 12288); 128-wide tiles are charged 10% more for their higher operand
// traffic per FLOP.
inline int pick_bn(int64_t M, int64_t N, int sms, unsigned allowed) {
    int best = 0;
    double best_cost = 0.0;
    for (int bn : {256, 192, 128}) {
        const unsigned bit = bn == 256 ? kBN256 : (bn == 192 ? kBN192 : kBN128);
        if (!(allowed & bit)) continue;
        const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);
        const int64_t waves = (tiles + sms - 1) / sms;
        const double cost = static_cast<double>(waves) * (bn + 96) * (bn == 128 ? 1.1 : 1.0);
        if (best == 0 || cost < best_cost - 1e-9) {
            best = bn;
            best_cost = cost;
        }
    }
    return best;
}

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

// D = A * B with the epilogue Epi, storing through the output tensors
// outs[0 .. num_out_maps<Epi>()) and reading the input tensor ins[0] (epilogues
// with inputs). Offsets shift the operands' coordinates inside their tensor
// maps (used to address one vocabulary chunk of E). Gated epilogues: N counts
// output columns, and the second half of each B tile starts b_gate_off
// columns (rows, K-major) after the first.
// With kChunk != kChunkNone, `chunks` holds that role's buffers (the role's
// own Operand/OutView gives its columns and row pitch; its pointer is unused).
template <typename ElemT, int BN, bool A_MN, bool B_MN, class Epi, int kChunk = kChunkNone>
tpce_status launch_gemm(const char *name, const Operand &a, const Operand &b, const OutView *outs,
                        const OutView *ins, int M, int N, int K, int a_off_mn, int a_off_k, int b_off_mn,
                        int b_off_k, const typename Epi::Params &ep, cudaStream_t stream, bool timed = true,
                        int b_gate_off = 0, const Chunks *chunks = nullptr) {
    using Cfg = KernelCfg<BN, Epi>;
    constexpr int kTileN = Epi::kGated ? BN / 2 : BN;
    using OutT = typename Epi::Out;
    constexpr bool kF32 = std::is_same<ElemT, float>::value;
    constexpr uint32_t kBoxK = kRowBytes / sizeof(ElemT);  // contraction elements per 128-byte row
    if (M <= 0 || N <= 0 || K <= 0) return TPCE_ERR_SHAPE;
    const int dt = kF32 ? 1 : 0;
    const int odt = std::is_same<OutT, float>::value ? 1 : 0;
    auto map_a = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return A_MN ? make_tmap(m, dt, p, a.cols, rows, a.ld, 64, 64) : make_tmap(m, dt, p, a.cols, rows, a.ld, kBoxK, kBM);
    };
    auto map_b = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return B_MN ? make_tmap(m, dt, p, b.cols, rows, b.ld, 64, 64)
                    : make_tmap(m, dt, p, b.cols, rows, b.ld, kBoxK, kTileN);
    };
    auto map_c = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return make_tmap(m, odt, p, outs[0].cols, rows, outs[0].ld, 32, 32, Stage<OutT>::kSwizzle);
    };
    ChunkSet<kChunk> cs;
    bool ok = kChunk == kChunkA   ? build_chunk_maps(cs, chunks, map_a)
              : kChunk == kChunkB ? build_chunk_maps(cs, chunks, map_b)
                                  : build_chunk_maps(cs, chunks, map_c);
    if (!ok) return fail(TPCE_ERR_INVALID, "bad sequence chunks for %s", name);
    CUtensorMap ta, tb, tc[2];
    if (kChunk == kChunkA)
        ta = cs.m[0];
    else
        ok = map_a(&ta, a.ptr, a.rows);
    if (kChunk == kChunkB)
        tb = cs.m[0];
    else
        ok = ok && map_b(&tb, b.ptr, b.rows);
    for (int k = 0; k < 2; ++k) {
        if (k == 0 && kChunk == kChunkC)
            tc[0] = cs.m[0];
        else if (k < num_out_maps<Epi>())
            ok = ok && make_tmap(&tc[k], odt, outs[k].ptr, outs[k].cols, outs[k].rows, outs[k].ld, 32, 32,
                                 Stage<OutT>::kSwizzle);
        else
            tc[k] = ta;  // unused by this epilogue
    }
    CUtensorMap tin = ta;  // unused unless the epilogue takes an input
    if (Epi::kIns > 0)
        ok = ok && ins && make_tmap(&tin, odt, ins[0].ptr, ins[0].cols, ins[0].rows, ins[0].ld, 32, 32,
                                    Stage<OutT>::kSwizzle);
    if (!ok) return fail(TPCE_ERR_CUDA, "cuTensorMapEncodeTiled rejected an operand of %s", name);

    GemmShape s;
    s.M = M;
    s.N = N;
    s.K = K;
    s.tiles_m = (M + kBM - 1) / kBM;
    s.tiles_n = (N + kTileN - 1) / kTileN;
    s.k_blocks = (K + static_cast<int>(kBoxK) - 1) / static_cast<int>(kBoxK);
    s.group_m = pick_group_m(s.tiles_m, kBM, K, sizeof(ElemT));
    s.run_len = 1;  // the one-CTA kernel walks single tiles
    s.unit_cols = s.tiles_n;
    s.a_off_mn = a_off_mn;
    s.a_off_k = a_off_k;
    s.b_off_mn = b_off_mn;
    s.b_off_k = b_off_k;
    s.b_gate_off = b_gate_off;
    s.full_units = s.tiles_m * s.tiles_n;  // the one-CTA kernel never splits its tail
    s.split = 1;
    s.tail_tiles = 0;
    s.partial = nullptr;
    s.tickets = nullptr;
    s.l2_hint = 0;
    s.debug_withhold = 0;

    auto kern = tc_gemm_kernel<ElemT, BN, A_MN, B_MN, Epi, kChunk>;
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
    kern<<<grid, 64 + 32 * Epi::kWarps, Cfg::kSmemBytes, stream>>>(ta, tb, tc[0], tc[1], tin, cs, s, ep, err);
    return check_launch(name, stream);
}

// The CTA-pair kernel (bf16 operands): a 256 x BN tile per cluster of two CTAs.
// Build-time switch: 256 (default) runs every bf16 GEMM on CTA pairs with
// 256 x 256 tiles; 0 keeps the one-CTA kernel (measured on GB300: the pair
// kernel is 10-12% faster, e.g. 1640 -> 1830 TFLOP/s on the 70B MLP step).
#ifndef TPCE_PAIR_BN
#define TPCE_PAIR_BN 256
#endif

// run_len > 1: each work unit is that many consecutive column tiles of one
// row-block (tiles_n must be a multiple of it; no split tail).
template <int BN, bool A_MN, bool B_MN, class Epi, int kChunk = kChunkNone>
tpce_status launch_gemm_pair(const char *name, const Operand &a, const Operand &b, const OutView *outs,
                             const OutView *ins, int M, int N, int K, int a_off_mn, int a_off_k, int b_off_mn,
                             int b_off_k, const typename Epi::Params &ep, cudaStream_t stream, bool timed = true,
                             int b_gate_off = 0, const Chunks *chunks = nullptr, const TailScratch *tail = nullptr,
                             int run_len = 1) {
    using Cfg = PairCfg<BN, Epi>;
    constexpr int kTileN = Epi::kGated ? BN / 2 : BN;
    using OutT = typename Epi::Out;
    if (M <= 0 || N <= 0 || K <= 0) return TPCE_ERR_SHAPE;
    const int odt = std::is_same<OutT, float>::value ? 1 : 0;
    auto map_a = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return A_MN ? make_tmap(m, 0, p, a.cols, rows, a.ld, 64, 64) : make_tmap(m, 0, p, a.cols, rows, a.ld, 64, kBM);
    };
    auto map_b = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return B_MN ? make_tmap(m, 0, p, b.cols, rows, b.ld, 64, 64) : make_tmap(m, 0, p, b.cols, rows, b.ld, 64, BN / 2);
    };
    auto map_c = [&](CUtensorMap *m, const void *p, int64_t rows) {
        return make_tmap(m, odt, p, outs[0].cols, rows, outs[0].ld, 32, 32, Stage<OutT>::kSwizzle);
    };
    ChunkSet<kChunk> cs;
    bool ok = kChunk == kChunkA   ? build_chunk_maps(cs, chunks, map_a)
              : kChunk == kChunkB ? build_chunk_maps(cs, chunks, map_b)
                                  : build_chunk_maps(cs, chunks, map_c);
    if (!ok) return fail(TPCE_ERR_INVALID, "bad sequence chunks for %s", name);
    CUtensorMap ta, tb, tc[2];
    if (kChunk == kChunkA)
        ta = cs.m[0];
    else
        ok = map_a(&ta, a.ptr, a.rows);
    if (kChunk == kChunkB)
        tb = cs.m[0];
    else
        ok = ok && map_b(&tb, b.ptr, b.rows);
    for (int k = 0; k < 2; ++k) {
        if (k == 0 && kChunk == kChunkC)
            tc[0] = cs.m[0];
        else if (k < num_out_maps<Epi>())
            ok = ok && make_tmap(&tc[k], odt, outs[k].ptr, outs[k].cols, outs[k].rows, outs[k].ld, 32, 32,
                                 Stage<OutT>::kSwizzle);
        else
            tc[k] = ta;
    }
    CUtensorMap tin = ta;  // unused unless the epilogue takes an input
    if (Epi::kIns > 0)
        ok = ok && ins && make_tmap(&tin, odt, ins[0].ptr, ins[0].cols, ins[0].rows, ins[0].ld, 32, 32,
                                    Stage<OutT>::kSwizzle);
    if (!ok) return fail(TPCE_ERR_CUDA, "cuTensorMapEncodeTiled rejected an operand of %s", name);
    GemmShape s;
    s.M = M;
    s.N = N;
    s.K = K;
    s.tiles_m = (M + 2 * kBM - 1) / (2 * kBM);
    s.tiles_n = (N + kTileN - 1) / kTileN;
    s.k_blocks = (K + 63) / 64;
    s.group_m = pick_group_m(s.tiles_m, 2 * kBM, K, 2);
    if (run_len < 1 || s.tiles_n % run_len != 0) return fail(TPCE_ERR_INVALID, "run of %d tiles for %s", run_len, name);
    s.run_len = run_len;
    s.unit_cols = s.tiles_n / run_len;
    s.a_off_mn = a_off_mn;
    s.a_off_k = a_off_k;
    s.b_off_mn = b_off_mn;
    s.b_off_k = b_off_k;
    s.b_gate_off = b_gate_off;
    s.l2_hint = pick_l2_hint(s.group_m, s.tiles_n, 2 * kBM, BN, K, 2);
    s.debug_withhold = take_debug_withhold();
    auto kern = tc_gemm_pair_kernel<BN, A_MN, B_MN, Epi, kChunk>;
    static std::mutex attr_mu;
    static bool attr_done[64] = {};
    tpce_status st = set_smem_attr(kern, Cfg::kSmemBytes, attr_done, attr_mu);
    if (st != TPCE_OK) return st;
    const int sms = num_sms();
    uint32_t *err = device_error_word();
    if (sms < 2 || err == nullptr) return fail(TPCE_ERR_CUDA, "device query failed (%s)", name);
    const int64_t units = static_cast<int64_t>(s.tiles_m) * s.unit_cols;
    const int clusters = static_cast<int>(std::min<int64_t>(units, sms / 2));
    bool memset_ok = true;
    plan_tail(s, clusters, BN, tail, stream, memset_ok);
    if (!memset_ok) return fail(TPCE_ERR_CUDA, "cudaMemsetAsync of the tail tickets (%s)", name);
    const int grid = 2 * clusters;
    KernelTimer timer(timed ? name : nullptr, stream);
    kern<<<grid, 64 + 32 * Epi::kWarps, Cfg::kSmemBytes, stream>>>(ta, tb, tc[0], tc[1], tin, cs, s, ep, err);
    return check_launch(name, stream);
}

// launch_gemm with the tile width chosen by pick_bn among `Allowed`.
template <typename ElemT, bool A_MN, bool B_MN, class Epi, unsigned Allowed, int kChunk = kChunkNone>
tpce_status launch_gemm_auto(const char *name, const Operand &a, const Operand &b, const OutView *outs,
                             const OutView *ins, int M, int N, int K, int a_off_mn, int a_off_k, int b_off_mn,
                             int b_off_k, const typename Epi::Params &ep, cudaStream_t stream, int b_gate_off = 0,
                             const Chunks *chunks = nullptr, const TailScratch *tail = nullptr) {
    static_assert(!Epi::kGated || (Allowed & kBN192) == 0, "gated tiles are 128 or 256 wide");
    if constexpr (TPCE_PAIR_BN != 0 && std::is_same<ElemT, __nv_bfloat16>::value && Epi::kWarps == 4) {
        return launch_gemm_pair<TPCE_PAIR_BN, A_MN, B_MN, Epi, kChunk>(name, a, b, outs, ins, M, N, K, a_off_mn,
                                                                      a_off_k, b_off_mn, b_off_k, ep, stream, true,
                                                                      b_gate_off, chunks, tail);
    } else {
        const int sms = num_sms();
        if (sms <= 0) return fail(TPCE_ERR_CUDA, "device query failed (%s)", name);
        const unsigned allowed = (Allowed & TPCE_BN_MASK) ? (Allowed & TPCE_BN_MASK) : Allowed;
        // a gated tile's accumulator spans twice its output columns
        const int bn = pick_bn(M, Epi::kGated ? 2 * static_cast<int64_t>(N) : N, sms, allowed);
        if constexpr ((Allowed & kBN256) != 0) {
            if (bn == 256)
                return launch_gemm<ElemT, 256, A_MN, B_MN, Epi, kChunk>(name, a, b, outs, ins, M, N, K, a_off_mn,
                                                                       a_off_k, b_off_mn, b_off_k, ep, stream, true,
                                                                       b_gate_off, chunks);
        }
        if constexpr ((Allowed & kBN192) != 0) {
            if (bn == 192)
                return launch_gemm<ElemT, 192, A_MN, B_MN, Epi, kChunk>(name, a, b, outs, ins, M, N, K, a_off_mn,
                                                                       a_off_k, b_off_mn, b_off_k, ep, stream, true,
                                                                       b_gate_off, chunks);
        }
        if constexpr ((Allowed & kBN128) != 0) {
            if (bn == 128)
                return launch_gemm<ElemT, 128, A_MN, B_MN, Epi, kChunk>(name, a, b, outs, ins, M, N, K, a_off_mn,
                                                                       a_off_k, b_off_mn, b_off_k, ep, stream, true,
                                                                       b_gate_off, chunks);
        }
        return fail(TPCE_ERR_SHAPE, "no tile width for %s", name);
    }
}

}  // namespace
}  // namespace tpce
