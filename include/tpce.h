/*
 * tpce.h -- C ABI of libtpce: Megatron-style 1D tensor-parallel MLP block and
 * vocabulary-parallel fused cross-entropy, with all t shards on one GPU.
 *
 * The partition follows "Tensor Parallelism and Pipeline Parallelism:
 * Mathematical Foundations of Megatron-LM 1D Slicing ..." (llms.blog),
 * sections "Column-Parallel Linear Layer", "Row-Parallel Linear Layer" and
 * "Conjugate Communication Operators", and "Cutting a Model Into Pieces"
 * (lecture 3), section "Megatron-LM: cutting inside the layer":
 *
 *   A = [A_1 .. A_t] split by columns, Y_i = GeLU(X A_i + bA_i) per shard
 *   with no exchange; B = [B_1; ..; B_t] split by rows, Z_i = Y_i B_i, and
 *   the forward operator g sums Z = sum_i Z_i (+ bB once). Backward: g*
 *   hands dZ to every shard unchanged, f* sums the per-shard dX_i.
 *
 * The fused logit GEMM + cross-entropy follows "LIT-022: Megatron-LM:
 * Training Multi-Billion Parameter Language Models Using Model Parallelism"
 * (anthology digest), "Key takeaways": each vocabulary shard reduces its
 * logits to per-token statistics, so b*s numbers are combined instead of
 * b*s*v logits. The vocabulary is padded to a multiple of 128 * t (same
 * bullet, and "Megatron-LM, in depth", section "Failure modes").
 *
 * On one GPU the shard index is a coordinate of the kernels' tile grid and
 * every sum over shards (g, f*, the statistics exchange, the dH sum) is done
 * on the device: in the tensor-core accumulator or in a reduction kernel.
 * There is no collective.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers owned by the caller; the
 *    library never allocates device memory and never frees a pointer.
 *  - Row-major layouts. X, Z, dX, dZ, H, dH: [T, h]. A, dA: [h, f].
 *    B, dB: [f, h]. U, Y (saved activations): [T, f]. E, dE: [v_pad, h].
 *    Shard i is the column block A[:, i f/t : (i+1) f/t], the row block
 *    B[i f/t : (i+1) f/t, :] and the row block E[i v_pad/t : (i+1) v_pad/t, :];
 *    the unsharded tensors are passed and t selects the partition.
 *  - dtype TPCE_BF16: X, A, B, Z, U, Y, dZ, dX, dA, dB, H, E, dH, dE are bf16,
 *    accumulation is fp32. dtype TPCE_F32: the same tensors are fp32 and the
 *    tensor cores read them as tf32 (10-bit mantissa), fp32 accumulate; this
 *    path stages transposed copies of some operands in the workspace. Biases
 *    and bias gradients are always fp32.
 *  - Every tensor pointer must be 16-byte aligned; h must be a multiple of 8.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream). Shape and alignment checks run on the host before any
 *    launch; a failed check launches nothing.
 *  - Gradients are written, not accumulated.
 *  - Errors are returned as tpce_status; nothing is thrown across the ABI.
 *    Problems only the device can see (a target id out of range, a bounded
 *    wait inside a kernel that ran out) are recorded in a device status word
 *    that tpce_device_status() reads.
 */
#ifndef TPCE_H
#define TPCE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TPCE_BF16 = 0,   /* bf16 tensors, fp32 accumulate */
    TPCE_F32 = 1     /* fp32 tensors, multiplied as tf32 on the tensor cores, fp32 accumulate */
} tpce_dtype;

/* Which dimension of a linear layer's weight W [n_in, n_out] the t shards
 * split ("Distributed tensor parallelism: scale fine-tuning of 70B-parameter
 * LLMs with Megatron-LM", section "The Mechanics of Tensor Parallelism (TP)
 * in Megatron-LM": ColumnParallelLinear and RowParallelLinear). */
typedef enum {
    TPCE_COLUMN_PARALLEL = 0,  /* W split by columns: n_out / t per shard */
    TPCE_ROW_PARALLEL = 1      /* W split by rows (X by columns): n_in / t per shard */
} tpce_parallel;

typedef enum {
    TPCE_OK = 0,
    TPCE_ERR_INVALID = 1,      /* null pointer, bad dtype, target id out of range */
    TPCE_ERR_SHAPE = 2,        /* sizes violate the partition rules */
    TPCE_ERR_ALIGN = 3,        /* a pointer is not 16-byte aligned */
    TPCE_ERR_WORKSPACE = 4,    /* workspace missing or smaller than the query says */
    TPCE_ERR_CUDA = 5,         /* a CUDA runtime/driver call failed */
    TPCE_ERR_TIMEOUT = 6,      /* a bounded wait inside a kernel gave up */
    TPCE_ERR_UNSUPPORTED = 7   /* valid request this build does not implement */
} tpce_status;

/* Human-readable name of a status. Never NULL. */
const char *tpce_status_string(tpce_status s);

/* Library ABI version (major * 100 + minor). */
int tpce_version(void);

/* Description of the last failure a call made on this host thread returned
 * (the failing CUDA call or check and its error name). Empty if none. The
 * text stays valid until the next failing call on the same thread. Setting
 * the environment variable TPCE_SYNC_CHECK=1 makes the library synchronise
 * after every kernel launch, so that an execution error is attributed to the
 * kernel that raised it (debugging aid; slow). */
const char *tpce_last_error(void);

/* ---------------------------------------------------------------------------
 * Vocabulary padding rule: the smallest multiple of divisor * t that is
 * >= v (divisor 128 is Megatron's default; 50,257 -> 51,200 at t = 8). Source:
 * LIT-022 digest, "Key takeaways" (vocabulary padded so each slice is a
 * multiple of 128); "Megatron-LM, in depth", "Failure modes" (rounded up to a
 * multiple of the divisor times TP). Returns -1 if v < 0, t < 1 or
 * divisor < 1.
 * ------------------------------------------------------------------------- */
int64_t tpce_pad_vocab(int64_t v, int t, int divisor);

/* ---------------------------------------------------------------------------
 * Workspace sizes in bytes (0 when none is needed). The caller allocates at
 * least this much device memory, 256-byte aligned, and passes it with its
 * size. The contents need not be initialised and are garbage afterwards.
 * tpce_mlp_workspace_bytes covers both tp_mlp_forward (which needs none) and
 * tp_mlp_backward. tpce_ce_workspace_bytes depends on whether gradients are
 * requested (with_grads != 0): the forward keeps per-token statistics only;
 * the backward adds a bounded bf16 scratch for one vocabulary chunk of
 * logit gradients and, when there is more than one chunk, an fp32 [T, h]
 * accumulator for dH. Returns 0 for invalid shapes.
 * ------------------------------------------------------------------------- */
size_t tpce_mlp_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype);
/* The optional workspace of the bf16 forward calls (tp_mlp_forward,
 * tp_swiglu_forward, tp_linear_forward, the attention forwards and their
 * sequence-parallel forms): with ws_bytes >= this, a GEMM whose last wave of
 * tiles is short splits those tiles along K over the idle SMs (each part's
 * fp32 partial written to the workspace, the last part summing them in part
 * order); with ws NULL the GEMMs run unsplit. Results differ only by the fp32
 * summation order of those tiles and are deterministic either way. Every
 * workspace query below includes this region at the start. */
size_t tpce_tail_workspace_bytes(void);
/* (the MLP query covers both calls of one dtype; TPCE_F32 adds transposed
 * copies of A, B, Y, dZ, X and dU) */
size_t tpce_ce_workspace_bytes(int64_t T, int64_t h, int64_t v_pad, int t, int dtype,
                               int with_grads);

/* ---------------------------------------------------------------------------
 * tp_mlp_forward -- the tensor-parallel MLP block, forward.
 *   U = X A + bA,  Y = GeLU(U)   (column-parallel GEMM1; per shard i the
 *                                 columns of A_i; GeLU needs no exchange)
 *   Z = sum_i Y_i B_i + bB       (row-parallel GEMM2; g = sum over shards,
 *                                 done in the accumulator; bB added once)
 * GeLU is the exact form x * Phi(x) (Phi via erf).
 * Inputs:  X [T, h], A [h, f], B [f, h]; bA [f] and bB [h] fp32, may be NULL
 *          (zero bias).
 * Outputs: Z [T, h]; U [T, f] and Y [T, f] are written for the backward.
 * Shapes:  T >= 0 (T == 0 is a no-op and every pointer may then be NULL),
 *          h >= 8 and h % 8 == 0, t >= 1, f % t == 0 and (f / t) % 64 == 0.
 * Workspace: none for TPCE_BF16 (ws may be NULL, ws_bytes 0); for TPCE_F32,
 *          tpce_mlp_workspace_bytes(T, h, f, t, TPCE_F32) bytes.
 * ------------------------------------------------------------------------- */
tpce_status tp_mlp_forward(const void *X, const void *A, const float *bA,
                           const void *B, const float *bB,
                           int64_t T, int64_t h, int64_t f, int t, int dtype,
                           void *Z, void *U, void *Y,
                           void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * tp_mlp_backward -- gradients of the block for the upstream gradient dZ.
 * Chain rule of tp_mlp_forward, with the conjugate operators of the
 * Mathematical Foundations page: g* gives dZ to every shard,
 *   dB_i = Y_i^T dZ,  dY_i = dZ B_i^T,  dU_i = dY_i (.) GeLU'(U_i),
 *   dA_i = X^T dU_i,  dbA_i = sum_tokens dU_i,  dbB = sum_tokens dZ,
 * and f* sums the shard partials  dX = sum_i dU_i A_i^T  (in the accumulator).
 * Inputs:  dZ [T, h], X [T, h], A [h, f], B [f, h], and the U [T, f] and
 *          Y [T, f] that tp_mlp_forward wrote for the same X, A, bA.
 * Outputs: dX [T, h], dA [h, f], dB [f, h]; dbA [f] and dbB [h] fp32, may be
 *          NULL (not computed).
 * Shapes:  as tp_mlp_forward. T == 0 writes zero weight/bias gradients; the
 *          token-dimension pointers (dZ, X, U, Y, dX) may then be NULL.
 * Workspace: tpce_mlp_workspace_bytes(T, h, f, t, dtype) bytes (holds dU).
 * ------------------------------------------------------------------------- */
tpce_status tp_mlp_backward(const void *dZ, const void *X, const void *A, const void *B,
                            const void *U, const void *Y,
                            int64_t T, int64_t h, int64_t f, int t, int dtype,
                            void *dX, void *dA, float *dbA, void *dB, float *dbB,
                            void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Sequence-parallel entry and exit ("Mathematical Foundations of Megatron-LM
 * 1D Slicing ...", section "Sequence Parallelism"). Outside the
 * tensor-parallel region each of the t ranks holds one sequence chunk of the
 * activations, rows [r T/t, (r+1) T/t). These calls take X, Z, dZ and dX as
 * t chunk buffers, one per rank:
 *   entry: the column-parallel GEMM reads the all-gathered X directly from
 *          the X chunks (and the backward reads the all-gathered dZ);
 *   exit:  the row-parallel GEMM's epilogue writes each shard-summed row of
 *          Z into the chunk that owns it -- the reduce-scatter -- and the
 *          backward writes dX the same way.
 * Every other tensor (A, B, biases, U, Y, the weight gradients) is as in
 * tp_mlp_forward / tp_mlp_backward, and so is the arithmetic: the results
 * are the rows of the dense calls' results, bit for bit.
 * Chunk arguments: host arrays of t device pointers, read during the call
 * only; chunk r is [T/t, h] row-major, 16-byte aligned.
 * Shapes: as the dense calls, and t <= 16, T % t == 0, (T / t) % 128 == 0
 * (whole 128-row tile blocks per chunk). T == 0: the forward is a no-op, the
 * backward zeroes the weight and bias gradients.
 * Workspace: as the dense calls.
 * ------------------------------------------------------------------------- */
tpce_status tp_mlp_forward_sp(const void *const *X_chunks, const void *A, const float *bA,
                              const void *B, const float *bB,
                              int64_t T, int64_t h, int64_t f, int t, int dtype,
                              void *const *Z_chunks, void *U, void *Y,
                              void *ws, size_t ws_bytes, void *stream);
tpce_status tp_mlp_backward_sp(const void *const *dZ_chunks, const void *const *X_chunks,
                               const void *A, const void *B, const void *U, const void *Y,
                               int64_t T, int64_t h, int64_t f, int t, int dtype,
                               void *const *dX_chunks, void *dA, float *dbA, void *dB, float *dbB,
                               void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * The SwiGLU variant of the block ("Distributed tensor parallelism: scale
 * fine-tuning of 70B-parameter LLMs with Megatron-LM", section "The MLP
 * Block"): MLP(X) = (Swish(X W_gate) (.) (X W_up)) W_down, with W_gate and
 * W_up column-parallel and W_down row-parallel. Swish(x) = x sigmoid(x).
 *
 * W1 = [W_gate | W_up] is one [h, 2f] matrix: columns 0..f-1 are the gate,
 * f..2f-1 the up projection. Shard i owns gate columns [i f/t, (i+1) f/t)
 * and the same range of up columns (f + i f/t ...), and rows [i f/t, ...) of
 * W2 = W_down [f, h]. b1 [2f] (gate biases, then up biases) and b2 [h] are
 * fp32 and may be NULL; b2 is added once, after the shard sum.
 *
 * tpce_swiglu_workspace_bytes covers both calls of one dtype (bf16: the
 * backward's [dG | dUp]; TPCE_F32 adds transposed copies of W1, W2, Y, dZ, X
 * and [dG | dUp]). Returns 0 for invalid shapes.
 * ------------------------------------------------------------------------- */
size_t tpce_swiglu_workspace_bytes(int64_t T, int64_t h, int64_t f, int t, int dtype);

/* ---------------------------------------------------------------------------
 * tp_swiglu_forward -- the SwiGLU block, forward.
 *   [G | Up] = X W1 + b1        (column-parallel GEMM1: each output tile
 *                                holds the gate and up columns of the same
 *                                shard columns; no exchange)
 *   Y = Swish(G) (.) Up
 *   Z = sum_i Y_i W2_i + b2     (row-parallel GEMM2; g = sum over shards, in
 *                                the accumulator)
 * Inputs:  X [T, h], W1 [h, 2f], W2 [f, h]; b1, b2 as above.
 * Outputs: Z [T, h]; GU = [G | Up] [T, 2f] and Y [T, f] are written for the
 *          backward.
 * Shapes:  as tp_mlp_forward (h >= 8, h % 8 == 0, f % t == 0,
 *          (f / t) % 64 == 0; T == 0 is a no-op, pointers may then be NULL).
 * Workspace: none for TPCE_BF16; for TPCE_F32,
 *          tpce_swiglu_workspace_bytes(T, h, f, t, TPCE_F32) bytes.
 * ------------------------------------------------------------------------- */
tpce_status tp_swiglu_forward(const void *X, const void *W1, const float *b1,
                              const void *W2, const float *b2,
                              int64_t T, int64_t h, int64_t f, int t, int dtype,
                              void *Z, void *GU, void *Y,
                              void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * tp_swiglu_backward -- gradients of the SwiGLU block for upstream dZ.
 * g* gives dZ to every shard:
 *   dW2_i = Y_i^T dZ,  dY_i = dZ W2_i^T,
 *   dG_i = dY_i (.) Up_i (.) Swish'(G_i),  dUp_i = dY_i (.) Swish(G_i),
 *   dW1 = X^T [dG | dUp],  db1 = sum_tokens [dG | dUp],  db2 = sum_tokens dZ,
 * and f* sums the shard partials  dX = sum_i [dG_i | dUp_i] W1_i^T  (in the
 * accumulator), Swish'(g) = s (1 + g (1 - s)), s = sigmoid(g).
 * Inputs:  dZ [T, h], X [T, h], W1 [h, 2f], W2 [f, h], and the GU [T, 2f]
 *          and Y [T, f] that tp_swiglu_forward wrote for the same X, W1, b1.
 * Outputs: dX [T, h], dW1 [h, 2f], dW2 [f, h]; db1 [2f] and db2 [h] fp32,
 *          may be NULL (not computed).
 * Shapes:  as tp_swiglu_forward. T == 0 writes zero weight/bias gradients.
 * Workspace: tpce_swiglu_workspace_bytes(T, h, f, t, dtype) bytes.
 * ------------------------------------------------------------------------- */
tpce_status tp_swiglu_backward(const void *dZ, const void *X, const void *W1, const void *W2,
                               const void *GU, const void *Y,
                               int64_t T, int64_t h, int64_t f, int t, int dtype,
                               void *dX, void *dW1, float *db1, void *dW2, float *db2,
                               void *ws, size_t ws_bytes, void *stream);

/* The sequence-parallel forms of the SwiGLU block: as tp_mlp_forward_sp /
 * tp_mlp_backward_sp, with the tensors of tp_swiglu_forward / backward. */
tpce_status tp_swiglu_forward_sp(const void *const *X_chunks, const void *W1, const float *b1,
                                 const void *W2, const float *b2,
                                 int64_t T, int64_t h, int64_t f, int t, int dtype,
                                 void *const *Z_chunks, void *GU, void *Y,
                                 void *ws, size_t ws_bytes, void *stream);
tpce_status tp_swiglu_backward_sp(const void *const *dZ_chunks, const void *const *X_chunks,
                                  const void *W1, const void *W2, const void *GU, const void *Y,
                                  int64_t T, int64_t h, int64_t f, int t, int dtype,
                                  void *const *dX_chunks, void *dW1, float *db1, void *dW2, float *db2,
                                  void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Linear layers: ColumnParallelLinear and RowParallelLinear ("Mathematical
 * Foundations of Megatron-LM 1D Slicing", sections "Column-Parallel Linear
 * Layer" and "Row-Parallel Linear Layer"). Both compute
 *   Y = X W + b,  X [T, n_in], W [n_in, n_out], b [n_out] fp32 or NULL,
 * and differ in where a shard sum falls (done in a GEMM accumulator here):
 *   TPCE_COLUMN_PARALLEL  forward: each shard's columns, no exchange;
 *                         backward: dX = sum_i dY_i W_i^T (f*).
 *   TPCE_ROW_PARALLEL     forward: Y = sum_i X_i W_i (g), b added once;
 *                         backward: each shard's columns of dX, no sum.
 * Backward: dX = dY W^T, dW = X^T dY, db = sum_tokens dY (db may be NULL).
 * Shapes: n_in, n_out >= 8 and multiples of 8; the split dimension (n_out for
 * column, n_in for row) divides by t into whole 64-wide blocks. T == 0: the
 * forward is a no-op, the backward zeroes dW and db.
 * Workspace: tpce_linear_workspace_bytes (bf16 forward: none; the backward
 * holds the bias-gradient partials; TPCE_F32 adds transposed copies of W, X
 * and dY). Returns 0 for invalid shapes.
 * ------------------------------------------------------------------------- */
size_t tpce_linear_workspace_bytes(int64_t T, int64_t n_in, int64_t n_out, int t, int parallel,
                                   int dtype);
tpce_status tp_linear_forward(const void *X, const void *W, const float *b,
                              int64_t T, int64_t n_in, int64_t n_out, int t, int parallel,
                              int dtype, void *Y, void *ws, size_t ws_bytes, void *stream);
tpce_status tp_linear_backward(const void *dY, const void *X, const void *W,
                               int64_t T, int64_t n_in, int64_t n_out, int t, int parallel,
                               int dtype, void *dX, void *dW, float *db,
                               void *ws, size_t ws_bytes, void *stream);

/* Sequence-parallel forms of the linear layers ("Mathematical Foundations ...",
 * section "Sequence Parallelism"), with the chunk conventions of
 * tp_mlp_forward_sp (host arrays of t device pointers, chunk r = rows
 * [r T/t, (r+1) T/t), (T / t) % 128 == 0, t <= 16):
 *   column-parallel entry: X as chunks (the GEMM reads the all-gathered X);
 *     the backward writes dX as chunks (the f* sum reduce-scattered);
 *   row-parallel exit: Y as chunks (the g sum reduce-scattered); the
 *     backward reads the gathered dY from its chunks.
 * Results are the rows of the dense calls' results. */
tpce_status tp_column_linear_forward_sp(const void *const *X_chunks, const void *W, const float *b,
                                        int64_t T, int64_t n_in, int64_t n_out, int t, int dtype,
                                        void *Y, void *ws, size_t ws_bytes, void *stream);
tpce_status tp_column_linear_backward_sp(const void *dY, const void *const *X_chunks, const void *W,
                                         int64_t T, int64_t n_in, int64_t n_out, int t, int dtype,
                                         void *const *dX_chunks, void *dW, float *db,
                                         void *ws, size_t ws_bytes, void *stream);
tpce_status tp_row_linear_forward_sp(const void *X, const void *W, const float *b,
                                     int64_t T, int64_t n_in, int64_t n_out, int t, int dtype,
                                     void *const *Y_chunks, void *ws, size_t ws_bytes, void *stream);
tpce_status tp_row_linear_backward_sp(const void *const *dY_chunks, const void *X, const void *W,
                                      int64_t T, int64_t n_in, int64_t n_out, int t, int dtype,
                                      void *dX, void *dW, float *db,
                                      void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Attention projections ("Distributed tensor parallelism ...", section "The
 * Multi-Head Attention Block"; "Mathematical Foundations ...", section
 * "Self-Attention Layer Decomposition"). The attention core between them is
 * not part of this library.
 *
 * tp_attn_qkv_*: the fused Q, K, V projection, column-parallel by heads:
 *   QKV = X Wqkv + bqkv,  X [T, h], Wqkv [h, (n_heads + 2 n_kv_heads) d],
 * columns grouped by key/value head g: the n_heads / n_kv_heads query heads
 * that share K_g and V_g, then K_g, then V_g (each head d wide), so that
 * shard i's contiguous column block holds whole groups: n_heads / t query
 * and n_kv_heads / t key/value heads (grouped-query attention; with 64 query
 * and 8 key/value heads at t = 8, 8 and 1 per shard). The backward's dX is
 * the f* sum over shards.
 * Shapes: n_heads % n_kv_heads == 0, n_kv_heads % t == 0, d >= 8, d % 8 == 0,
 * and a shard's (n_heads + 2 n_kv_heads) d / t columns are whole 64-wide
 * blocks; the rest as tp_linear_* with n_in = h.
 *
 * tp_attn_out_*: the output projection W_O, row-parallel over the
 * concatenated head outputs O [T, n_heads d]:  Z = sum_i O_i W_O,i + bo,
 * Wo [n_heads d, h]; n_heads % t == 0 and n_heads d / t whole 64-wide blocks.
 *
 * tpce_attn_workspace_bytes covers all four calls of one dtype.
 * ------------------------------------------------------------------------- */
size_t tpce_attn_workspace_bytes(int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                 int64_t head_dim, int t, int dtype);
tpce_status tp_attn_qkv_forward(const void *X, const void *Wqkv, const float *bqkv,
                                int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                int64_t head_dim, int t, int dtype, void *QKV,
                                void *ws, size_t ws_bytes, void *stream);
tpce_status tp_attn_qkv_backward(const void *dQKV, const void *X, const void *Wqkv,
                                 int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                 int64_t head_dim, int t, int dtype,
                                 void *dX, void *dWqkv, float *dbqkv,
                                 void *ws, size_t ws_bytes, void *stream);
tpce_status tp_attn_out_forward(const void *O, const void *Wo, const float *bo,
                                int64_t T, int64_t h, int64_t n_heads, int64_t head_dim, int t,
                                int dtype, void *Z, void *ws, size_t ws_bytes, void *stream);
tpce_status tp_attn_out_backward(const void *dZ, const void *O, const void *Wo,
                                 int64_t T, int64_t h, int64_t n_heads, int64_t head_dim, int t,
                                 int dtype, void *dO, void *dWo, float *dbo,
                                 void *ws, size_t ws_bytes, void *stream);

/* Sequence-parallel forms of the attention projections: the QKV projection
 * is the column-parallel entry (X and dX as chunks), the output projection
 * the row-parallel exit (Z and dZ as chunks); chunk rules as above. */
tpce_status tp_attn_qkv_forward_sp(const void *const *X_chunks, const void *Wqkv, const float *bqkv,
                                   int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                   int64_t head_dim, int t, int dtype, void *QKV,
                                   void *ws, size_t ws_bytes, void *stream);
tpce_status tp_attn_qkv_backward_sp(const void *dQKV, const void *const *X_chunks, const void *Wqkv,
                                    int64_t T, int64_t h, int64_t n_heads, int64_t n_kv_heads,
                                    int64_t head_dim, int t, int dtype,
                                    void *const *dX_chunks, void *dWqkv, float *dbqkv,
                                    void *ws, size_t ws_bytes, void *stream);
tpce_status tp_attn_out_forward_sp(const void *O, const void *Wo, const float *bo,
                                   int64_t T, int64_t h, int64_t n_heads, int64_t head_dim, int t,
                                   int dtype, void *const *Z_chunks, void *ws, size_t ws_bytes,
                                   void *stream);
tpce_status tp_attn_out_backward_sp(const void *const *dZ_chunks, const void *O, const void *Wo,
                                    int64_t T, int64_t h, int64_t n_heads, int64_t head_dim, int t,
                                    int dtype, void *dO, void *dWo, float *dbo,
                                    void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * vocab_parallel_ce -- logit GEMM fused with softmax cross-entropy, the
 * vocabulary split into t shards of v_pad / t rows of E.
 * Forward, per shard i and token r (the logits l = H E_i^T stay in fp32
 * registers and are never written to memory):
 *   m_i = max of l over the shard's real ids (< v_valid),
 *   s_i = sum exp(l - m_i) over them, tau = l[target] in the owning shard.
 * Only (m_i, s_i) and tau are combined across shards:
 *   m = max_i m_i,  S = sum_i s_i exp(m_i - m),  lse = m + ln S,
 *   loss = lse - tau.
 * The logit GEMM reaches each shard's (m_i, s_i) through p_i partial pairs
 * per token, each the fold over one run of consecutive vocabulary tiles;
 * where p_i > 1 the epilogue that finishes a shard's last run folds them, so
 * the combine reads exactly one pair per shard and token. p_i = 1 when the
 * GEMM's work units fill the GPU in one wave, else the fewest equal parts
 * that keep it evenly busy (9 for 16,384 tokens over 129,024 ids and t = 8;
 * one per 128-id tile for fp32).
 * Backward (dH and/or dE requested), with dl = grad_scale * (softmax - onehot)
 * on real ids and 0 on padded ids, recomputing the logits chunk by chunk:
 *   dE_i = dl_i^T H   (each shard's own rows, no exchange; padded rows = 0)
 *   dH   = sum_i dl_i E_i   (sum over shards on the device)
 * grad_scale is the upstream dLoss per token (1 for the sum, 1/T for the mean).
 * Inputs:  H [T, h], E [v_pad, h], targets [T] int32 in [0, v_valid).
 * Outputs: loss [T] fp32; lse [T] fp32 may be NULL; dH [T, h] and dE
 *          [v_pad, h] may be NULL (a NULL pair is the forward-only call).
 * Shapes:  T >= 0, h % 8 == 0, t >= 1, v_pad % t == 0, (v_pad / t) % 128 == 0,
 *          1 <= v_valid <= v_pad. T == 0 writes dE = 0 (if requested); H,
 *          targets and loss may then be NULL.
 * Errors:  a target outside [0, v_valid) gives a NaN loss for that token and
 *          TPCE_ERR_INVALID in the device status word.
 * Workspace: tpce_ce_workspace_bytes(T, h, v_pad, t, dtype, dH||dE) bytes.
 * ------------------------------------------------------------------------- */
tpce_status vocab_parallel_ce(const void *H, const void *E, const int32_t *targets,
                              int64_t T, int64_t h, int64_t v_pad, int64_t v_valid, int t,
                              float grad_scale, int dtype,
                              float *loss, float *lse, void *dH, void *dE,
                              void *ws, size_t ws_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * vocab_parallel_ce_loss_static -- the forward of vocab_parallel_ce (loss and
 * optionally lse, no gradients) that allocates nothing and needs no
 * workspace. The pages have no counterpart to this call; it exists for
 * callers that cannot call cudaMalloc, such as a plugin inside a host
 * framework whose memory planner owns every device buffer and forbids
 * allocations it did not plan, or a latency-critical path that must not risk
 * the implicit device synchronisation of an allocation.
 * The caller passes inputs and outputs exactly as for vocab_parallel_ce with
 * dH = dE = NULL. The per-token statistics live instead in a static device
 * array of TPCE_CE_STATIC_SCRATCH_BYTES bytes inside the library, which every
 * GPU that loads the library holds until the process exits. It must hold the
 * shards' pairs, t * T * 8 bytes; where shards are cut into parts (p_i > 1)
 * also the parts' pairs, (sum_i p_i) * T * 8 bytes, and ceil(T / 32) * t * 4
 * bytes of tickets; and T * 4 bytes of target logits (plus another T * 4 when
 * lse is NULL), each rounded up to 256 -- 10.6 MB for 16,384 tokens over
 * 129,024 ids at t = 8. Larger requests return TPCE_ERR_WORKSPACE with the
 * sizes in tpce_last_error(), before any launch.
 * The first call on a device, with that device current, looks up the array's
 * device address (cudaGetSymbolAddress) and caches it. Under CUDA's default
 * lazy module loading that first call is also when the array's memory is
 * committed on the device (under eager loading: when the library loads), a
 * one-time implicit allocation that fails if the device is full. Make the
 * first call per device before a memory planner reserves the device and
 * before any stream capture; later calls allocate nothing. All calls share the one array and it keeps the
 * last call's contents: a call writes every statistic it reads and clears
 * the tickets (a memset on its stream) before using them; calls whose kernels
 * overlap on the GPU race on it, so order them on one stream or with events.
 * Errors as vocab_parallel_ce.
 * ------------------------------------------------------------------------- */
#define TPCE_CE_STATIC_SCRATCH_BYTES (16u << 20)

tpce_status vocab_parallel_ce_loss_static(const void *H, const void *E, const int32_t *targets,
                                          int64_t T, int64_t h, int64_t v_pad, int64_t v_valid,
                                          int t, int dtype, float *loss, float *lse, void *stream);

/* ---------------------------------------------------------------------------
 * Device status word. Kernels record the first device-side failure (a
 * TPCE_ERR_* code in the low 8 bits, detail above) instead of trapping.
 * tpce_device_status synchronises `stream`, reads the word of the current
 * device, clears it when clear != 0, and returns its status code
 * (TPCE_ERR_CUDA if the synchronisation itself fails). *detail, if not NULL,
 * receives the raw word.
 * ------------------------------------------------------------------------- */
tpce_status tpce_device_status(void *stream, int clear, uint32_t *detail);

/* ---------------------------------------------------------------------------
 * Failure-path test knob (not for production use). The pages' in-depth
 * Megatron-LM page ("Megatron-LM, in depth", "Failure modes") treats a hung
 * collective as a failure to be detected rather than waited out; here every
 * wait inside a kernel is bounded, and this call lets a test make one wait
 * run out on purpose. tpce_debug_withhold_next_load(1) arms it: the next
 * bf16 GEMM launch on the CTA-pair kernel (any entry point) then arms the
 * full-barrier of its first pipeline stage in cluster 0 but issues none of
 * that stage's TMA loads, so the MMA thread's wait for it can never complete.
 * After its bound (2 s) that wait records TPCE_ERR_TIMEOUT (detail: which
 * wait, bits 8..) in the device status word and raises the CTA's abort flag;
 * the kernel's other waits then give up too (each bounded), in-flight loads
 * and stores land, tensor memory is freed and the kernel returns, leaving the
 * context usable. That launch's outputs are undefined. The arming is used up
 * by that one launch; tpce_debug_withhold_next_load(0) disarms it unused.
 * Process-wide; returns TPCE_OK.
 * ------------------------------------------------------------------------- */
tpce_status tpce_debug_withhold_next_load(int on);

/* ---------------------------------------------------------------------------
 * Kernel timing. While enabled, every kernel the library launches is
 * bracketed by two CUDA events recorded on the launch stream.
 * tpce_profile_enable(1) starts a fresh record (0 stops recording).
 * tpce_profile_count() waits for the recorded events, aggregates them by
 * kernel name and returns the number of distinct names (-1 on error).
 * tpce_profile_get(i, ...) returns entry i of that aggregate: the kernel's
 * name (static storage), number of launches and total milliseconds.
 * ------------------------------------------------------------------------- */
tpce_status tpce_profile_enable(int on);
int tpce_profile_count(void);
tpce_status tpce_profile_get(int i, const char **name, int64_t *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* TPCE_H */
