/*
 * tpmlp -- the tensor-parallel (Megatron-style) MLP block on one GB300 (sm_103a).
 *
 * The block (千亿参数模型如何拆分到多张GPU上训练, "方案一：按列切分权重矩阵" and
 * "方案二：按行切分权重矩阵"; 大模型分布式并行策略详解：TP、DP、PP、CP、EP核心原理与实战 §4.1;
 * AI大模型分布式训练：张量并行与流水线并行深度实践 §2.1-2.2):
 *
 *     Y_i = GeLU(X W1_i + b1_i)            i = 0..k-1, W1_i = W1[:, i f:(i+1) f]
 *     Z   = sum_i Y_i W2_i + b2                        W2_i = W2[i f:(i+1) f, :]
 *
 * with X [B, S, H], W1 [H, F], W2 [F, H], F = 4H on the pages' models (any F works),
 * f = F / k the shard width, and GeLU the exact erf form. The pages run each shard on
 * its own GPU and add the k partials with one All-Reduce; here all k shards run on one
 * GPU and the sum over shards is accumulated in the same fp32 tensor-memory tile of the
 * second GEMM, so it costs no extra pass over memory and no collective.
 *
 * Conventions for every call:
 *  - Pointers named "device" are CUDA device addresses on the context's device; the
 *    caller owns them and keeps them alive until the stream work that uses them is done.
 *  - Tensors are dense, row-major, bfloat16 unless stated otherwise; device pointers must
 *    be 16-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). All
 *    device work is enqueued on it; no call synchronises unless its comment says so.
 *  - A context belongs to the device that was current when it was created. Every call that
 *    enqueues work or touches the context's device memory first checks that this device is
 *    current on the calling thread and returns TPMLP_ERR_INVALID_ARG otherwise (nothing is
 *    launched; tpmlp_last_error names both devices).
 *  - Every call returns TPMLP_OK (0) or a negative tpmlp_status; no C++ exception or abort
 *    ever crosses this interface. A failed call leaves the context usable unless it
 *    returned TPMLP_ERR_CUDA (a sticky CUDA error, after which the context should be
 *    destroyed).
 *  - A context is used from one host thread at a time, and its GEMM calls on one stream at a
 *    time: calls on different streams must not overlap on the GPU, because they share the
 *    context's intermediate and split-reduction workspaces. Separate contexts are
 *    independent.
 *  - The GEMM kernels are launched with programmatic stream serialisation: each may be
 *    scheduled while the kernel before it in the stream finishes, and waits (griddepcontrol)
 *    for that kernel's results before touching global memory. Each also lets the next
 *    kernel in the stream be scheduled early. A kernel launched normally after a library call
 *    is unaffected. A caller's own kernel that is launched with programmatic stream
 *    serialisation after a library call must execute griddepcontrol.wait before it reads
 *    that call's outputs, as the programmatic dependent launch rules require anyway.
 */
#ifndef TPMLP_H
#define TPMLP_H

#include <stdint.h>

#if defined(__GNUC__)
#define TPMLP_API __attribute__((visibility("default")))
#else
#define TPMLP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct tpmlp_ctx tpmlp_ctx; /* opaque, owned by the library */

typedef enum {
    TPMLP_OK = 0,
    TPMLP_ERR_INVALID_ARG = -1,       /* null pointer, non-positive size, ... */
    TPMLP_ERR_UNSUPPORTED_SHAPE = -2, /* see tpmlp_create's shape rules */
    TPMLP_ERR_NOT_PACKED = -3,        /* forward before tpmlp_pack_shards */
    TPMLP_ERR_CUDA = -4,              /* a CUDA runtime/driver call failed (see tpmlp_last_error) */
    TPMLP_ERR_OOM = -5,               /* device allocation failed */
    TPMLP_ERR_DEVICE_TIMEOUT = -6,    /* a kernel gave up waiting on a pipeline barrier */
    TPMLP_ERR_ARCH = -7,              /* the current device is not sm_103 */
    TPMLP_ERR_MISALIGNED = -8         /* a device pointer is not 16-byte aligned */
} tpmlp_status;

/* Flags for tpmlp_create. */
#define TPMLP_FLAG_Z_FP32 0x1u    /* Z is written as fp32 instead of bf16 */
#define TPMLP_FLAG_SINGLE_SM 0x2u /* use only the single-SM kernel (128-row tiles), never the
                                     CTA-pair kernel (256 x 256 tiles on two SMs) */
#define TPMLP_FLAG_SWIGLU 0x4u    /* gated block: Y_i = SiLU(X Wg_i + bg_i) * (X Wu_i + bu_i);
                                     weights come from tpmlp_pack_shards_swiglu */
#define TPMLP_FLAG_FIXED_ORDER 0x8u /* never split an output tile's reduction across CTA pairs.
                                     By default, when the last wave of 256 x 256 tiles would
                                     leave CTA pairs idle, or a launch has fewer tiles than
                                     pairs (a small batch), the reductions of those tiles are
                                     divided among several pairs and their fp32 partial sums
                                     added in a fixed order; and in deep second GEMMs every
                                     second round of 512 x 256 units sums its reduction blocks
                                     last to first (the blocks still in L2 first). Results are
                                     deterministic, but their last bits then depend on the token
                                     count M. With this flag every tile is summed in one pass in
                                     reduction order, so the pair and single-SM kernels, and any
                                     M, give identical bits */

/*
 * Create a context for one block shape on the current CUDA device.
 *   out      receives the context (set to NULL on failure)
 *   H        hidden size (columns of X and Z); a multiple of 64
 *   F        intermediate size (columns of W1, rows of W2); a multiple of 64
 *   k        shard count: F % k == 0 and f = F/k a multiple of 64 (the pages' tensor
 *            parallel degree; shards are contiguous, equal column blocks of W1 and the
 *            matching row blocks of W2 -- AI大模型分布式训练 §2.1 splits W into
 *            [hidden, ffn/k] pieces)
 *   flags    0, or any of TPMLP_FLAG_Z_FP32, TPMLP_FLAG_SINGLE_SM, TPMLP_FLAG_SWIGLU,
 *            TPMLP_FLAG_FIXED_ORDER
 * Allocates the packed-weight buffers (2*H*F bf16 + (F+H) fp32), a device status word and,
 * unless TPMLP_FLAG_SINGLE_SM or TPMLP_FLAG_FIXED_ORDER is given, the split-reduction
 * workspace (two 128 KB slots of fp32 partial sums per CTA, 512 KB per CTA pair, plus
 * 64 bytes of arrival counters per SM: about 40 MB on 152 SMs); the intermediate activation
 * buffer is allocated by tpmlp_reserve or the first forward.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, ARCH (device is not sm_103), OOM, CUDA.
 */
TPMLP_API int tpmlp_create(tpmlp_ctx **out, int64_t H, int64_t F, int32_t k, uint32_t flags);

/*
 * Pack the weights into the kernels' layout (one-time per weight set; the shard packer).
 *   W1 device bf16 [H, F]   b1 device bf16 [F]   W2 device bf16 [F, H]   b2 device bf16 [H]
 * W1 is in the pages' math orientation (Y = X W1, AI大模型分布式训练 §2.1 allocates the
 * column-parallel weight as [in_features, out_features / k]), not [out, in].
 * Writes W1p [k][f][H] (each column shard transposed so that its reduction dimension H is
 * contiguous), W2p [k][H][f] (each row shard transposed likewise; in 16 KB blocks of 128 rows
 * x 64 columns when the second GEMM runs on CTA pairs, see tpmlp_packed_buffer), and fp32
 * copies of b1 and b2. The raw weights may be freed once the stream has passed this call.
 * Errors: INVALID_ARG (also: context created with TPMLP_FLAG_SWIGLU), MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_pack_shards(tpmlp_ctx *ctx, const void *W1, const void *b1, const void *W2,
                      const void *b2, void *stream);

/*
 * Pack the weights of the gated block (context created with TPMLP_FLAG_SWIGLU). The pages'
 * Llama-style feed-forward splits gate_up_proj by columns and down_proj by rows
 * (大模型分布式优化技术（一） §5.1; AI大模型分布式训练 §6.1: gate_proj / up_proj ColwiseParallel,
 * down_proj RowwiseParallel); the activation is SwiGLU (same first page, §3.3):
 *     Y_i = SiLU(X Wg_i + bg_i) * (X Wu_i + bu_i),   Z = sum_i Y_i W2_i + b2,
 *     SiLU(a) = a / (1 + e^-a), shard i = columns [i f, (i+1) f) of Wg and Wu.
 *   Wg, Wu device bf16 [H, F]   bg, bu device bf16 [F] (zeros for bias-free models)
 *   W2 device bf16 [F, H]       b2 device bf16 [H]
 * Writes one K-major operand holding both projections, interleaved in blocks of G = 128
 * (64 if f is not a multiple of 128) rows per shard, so that every tile of the first GEMM
 * holds the gate and up columns of the same outputs; W2 and b2 are packed as in
 * tpmlp_pack_shards. tpmlp_forward / tpmlp_gemm1 / tpmlp_gemm2 then run the gated block.
 * Errors: INVALID_ARG (also: context not created with TPMLP_FLAG_SWIGLU), MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_pack_shards_swiglu(tpmlp_ctx *ctx, const void *Wg, const void *bg,
                                       const void *Wu, const void *bu, const void *W2,
                                       const void *b2, void *stream);

/*
 * Make sure the intermediate buffer Y [M, F] (bf16) holds at least max_tokens rows.
 * Synchronises the device when it has to grow the buffer. Forward calls grow it on demand;
 * call this first to keep allocation out of a timed or captured region.
 * Errors: INVALID_ARG, OOM, CUDA.
 */
TPMLP_API int tpmlp_reserve(tpmlp_ctx *ctx, int64_t max_tokens);

/*
 * The block's forward pass: Z = sum_i GeLU(X W1_i + b1_i) W2_i + b2.
 *   X   device bf16 [B, S, H] (M = B*S token rows, each independent)
 *   Z   device [B, S, H], bf16 (or fp32 with TPMLP_FLAG_Z_FP32); must not overlap X
 * Two kernel launches on `stream`: the first GEMM with its fused bias + GeLU epilogue
 * writing Y [M, F] bf16 into the context's buffer, then the second GEMM, which sums all k
 * shards' partials in one fp32 accumulator and adds b2 once. B*S == 0 is a no-op (X and
 * Z may then be NULL).
 * Errors: INVALID_ARG, NOT_PACKED, MISALIGNED, OOM (growing Y), CUDA. A pipeline timeout
 * inside a kernel is reported by tpmlp_get_status, not here.
 * CUDA graphs: the call can be captured once tpmlp_reserve has sized Y for the captured token
 * count (capture forbids the allocation). Launches enqueued under stream capture never split
 * their reduction across CTA pairs, so a replay computes what an eager call with
 * TPMLP_FLAG_FIXED_ORDER computes.
 */
TPMLP_API int tpmlp_forward(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S, void *Z, void *stream);

/*
 * tpmlp_forward that also records the caller's CUDA event `after_gemm1` (a cudaEvent_t passed
 * as void*) on `stream` between the two kernel launches, so that each kernel can be timed
 * (cudaEventElapsedTime against events recorded before and after the call). No counterpart on
 * the pages. The same kernels, layouts and results as tpmlp_forward; the event costs the
 * overlap of the two launches (a few microseconds). Errors: as tpmlp_forward, plus
 * INVALID_ARG for a NULL event and CUDA if recording it fails.
 */
TPMLP_API int tpmlp_forward_marked(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S, void *Z,
                                   void *after_gemm1, void *stream);

/*
 * tpmlp_forward on host buffers: X (host, [B,S,H] bf16) in, Z (host, [B,S,H]) out; returns
 * once Z is in host memory (it waits for `stream`). Token rows are independent, so the work
 * streams in up to 4 row chunks: the copies of X chunks into a device staging buffer and of Z
 * chunks out of one run on two copy streams of the context and overlap the GEMMs of the other
 * chunks, which run on `stream` after the work already queued there. The chunk sizes are
 * planned once per token count under a pipeline model of the copies and of the GEMMs' rounds
 * of tiles (small end chunks, tile counts that fill whole rounds). Page-locked host memory
 * gives asynchronous, full-speed copies; pageable memory works but is slower.
 * Staging buffers are owned by the context and grow on demand. Not for stream capture: while
 * `stream` is capturing it returns INVALID_ARG and queues nothing.
 * Errors: as tpmlp_forward.
 */
TPMLP_API int tpmlp_forward_host(tpmlp_ctx *ctx, const void *X_host, int64_t B, int64_t S, void *Z_host,
                       void *stream);

/*
 * tpmlp_forward on host buffers without waiting: queues the copy of X_host in, the forward,
 * and the copy of Z out to Z_host, and returns. For a stream of calls (a serving loop): the
 * context stages each call in one of two device slots in turn, so a call's input copy runs
 * during the kernels of the call before it and its output copy during those of the call
 * after it. The kernels run on `stream` after the work already queued there; the copies run
 * on the context's two copy streams, ordered against the kernels by events. The whole call is
 * one chunk (no row-chunk plan: in a run of calls the copies are hidden by the neighbours'
 * kernels, and one full-size launch per GEMM is the fastest). Results equal tpmlp_forward's
 * for the same token count, bit for bit.
 *   X_host, Z_host  host bf16 [B,S,H] and [B,S,H] (fp32 with TPMLP_FLAG_Z_FP32). Both stay
 *                   owned by the caller and must stay valid, X_host unchanged and Z_host
 *                   unread, until tpmlp_host_wait returns. Buffers of calls in flight at the
 *                   same time must not overlap. Page-locked memory gives the overlap;
 *                   pageable memory works but each copy then blocks the host.
 * A larger token count than any earlier async call's waits for the device once (the slots
 * grow). Not for stream capture (INVALID_ARG, nothing queued).
 * Errors: as tpmlp_forward_host; a returned error leaves the calls queued before it
 * intact (tpmlp_host_wait still waits for them).
 */
TPMLP_API int tpmlp_forward_host_async(tpmlp_ctx *ctx, const void *X_host, int64_t B, int64_t S,
                                       void *Z_host, void *stream);

/*
 * Waits on the host until every host-buffer call of this context queued so far (the async
 * ones included) has written its Z to host memory. Errors: INVALID_ARG (NULL ctx), the device
 * check of every entry point, CUDA (a failed copy or kernel; the device status word, read by
 * tpmlp_get_status, tells a kernel's timeout apart).
 */
TPMLP_API int tpmlp_host_wait(tpmlp_ctx *ctx);

/*
 * The first step alone (column-parallel GEMM of every shard + b1 + GeLU):
 *   Y[m, i f + j] = GeLU(b1[i f + j] + sum_h X[m, h] W1[h, i f + j])   rounded to bf16
 *   X device bf16 [M, H]; Y device bf16 [M, F] (shard i in columns [i f, (i+1) f)).
 * M == 0 is a no-op (pointers may then be NULL).
 * Errors: INVALID_ARG, NOT_PACKED, MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_gemm1(tpmlp_ctx *ctx, const void *X, int64_t M, void *Y, void *stream);

/*
 * The second step alone (row-parallel GEMM of every shard, the sum over shards -- the
 * pages' All-Reduce -- done in the fp32 accumulator, + b2):
 *   Z[m, n] = b2[n] + sum_i sum_{j<f} Y[m, i f + j] W2[i f + j, n]
 *   Y device bf16 [M, F]; Z device [M, H] (bf16, or fp32 with TPMLP_FLAG_Z_FP32).
 * M == 0 is a no-op (pointers may then be NULL).
 * Errors: INVALID_ARG, NOT_PACKED, MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_gemm2(tpmlp_ctx *ctx, const void *Y, int64_t M, void *Z, void *stream);

/*
 * LayerNorm parameters for the layer around the block (see tpmlp_block_forward), or for the
 * input of a column-parallel linear layer (LayerNorm before the Q/K/V projection); the
 * normalised width is the block's H, or the layer's K. Not for row-parallel layers.
 *   gamma, beta  device bf16 [H] (copied; may be freed once the stream has passed this call)
 *   eps          0 <= eps <= 1, added to the variance inside the square root
 * H must be at most 16384 for the LayerNorm kernel.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, MISALIGNED, OOM, CUDA.
 */
TPMLP_API int tpmlp_set_layernorm(tpmlp_ctx *ctx, const void *gamma, const void *beta, float eps,
                                  void *stream);

/*
 * LayerNorm of each token's full hidden vector (the step in front of the block:
 * 大模型分布式并行策略详解 §4.2 -- LayerNorm needs the whole hidden state; sequence parallelism
 * splits it along the independent tokens, AI大模型分布式训练 §4.2):
 *   Xn[m, h] = (X[m, h] - mu_m) / sqrt(var_m + eps) * gamma[h] + beta[h]
 *   mu_m = mean_h X[m, h], var_m = mean_h (X[m, h] - mu_m)^2 (biased); fp32 statistics.
 *   X, Xn device bf16 [M, H]; M == 0 is a no-op.
 * Errors: INVALID_ARG, NOT_PACKED (parameters not set), MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_layernorm(tpmlp_ctx *ctx, const void *X, int64_t M, void *Xn, void *stream);

/*
 * The block inside its Transformer layer: Z = X + MLP(LayerNorm(X)) -- the residual add of the
 * pages' TransformerBlock (x = x + mlp(x), AI大模型分布式训练 §3.4) with LayerNorm in front.
 * MLP is the context's block (GeLU, or gated with TPMLP_FLAG_SWIGLU). Three launches: the
 * LayerNorm kernel, the first GEMM on the normalised input, and the second GEMM whose
 * epilogue adds X (Z = X + (sum_i Y_i W2_i + b2), in fp32, rounded once).
 *   X device bf16 [B, S, H]; Z device [B, S, H] (bf16, or fp32 with TPMLP_FLAG_Z_FP32).
 *   Z may be X itself (in-place update of the residual stream, bf16 output); no other
 *   overlap is allowed. The normalised input lives in a context buffer (grows on demand,
 *   synchronising the device when it does).
 * Errors: INVALID_ARG, NOT_PACKED (weights or LayerNorm parameters not set), MISALIGNED,
 * UNSUPPORTED_SHAPE, OOM, CUDA.
 */
TPMLP_API int tpmlp_block_forward(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S, void *Z,
                                  void *stream);

/*
 * tpmlp_block_forward on host buffers: X (host, [B,S,H] bf16) in, Z = X + MLP(LayerNorm(X))
 * (host, [B,S,H]) out; returns once Z is in host memory (it waits for `stream`). The same
 * row-chunk pipeline as tpmlp_forward_host: per chunk the LayerNorm kernel, the first GEMM and
 * the second GEMM with the residual add run on `stream` while the copies of the other chunks
 * in and out run on the context's copy streams. Z_host may equal X_host (the residual stream
 * updated in place). Requires tpmlp_set_layernorm.
 * Errors: as tpmlp_block_forward.
 */
TPMLP_API int tpmlp_block_forward_host(tpmlp_ctx *ctx, const void *X_host, int64_t B, int64_t S,
                                       void *Z_host, void *stream);

/*
 * tpmlp_block_forward_host without waiting, as tpmlp_forward_host_async is to
 * tpmlp_forward_host: the LayerNorm kernel, the first GEMM and the second GEMM with the
 * residual add of one call run on `stream` while the neighbouring calls' copies run; Z_host
 * may equal X_host within one call. Requires tpmlp_set_layernorm.
 * Errors: as tpmlp_block_forward_host.
 */
TPMLP_API int tpmlp_block_forward_host_async(tpmlp_ctx *ctx, const void *X_host, int64_t B,
                                             int64_t S, void *Z_host, void *stream);

/*
 * tpmlp_block_forward with the caller's CUDA events `after_layernorm` and `after_gemm1`
 * recorded on `stream` after the first and the second of its three launches (per-kernel
 * timing; see tpmlp_forward_marked). Errors: as tpmlp_block_forward, plus INVALID_ARG for a
 * NULL event and CUDA if recording one fails.
 */
TPMLP_API int tpmlp_block_forward_marked(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S,
                                         void *Z, void *after_layernorm, void *after_gemm1,
                                         void *stream);

/*
 * The second step with the residual add (the last launch of tpmlp_block_forward):
 *   Z[m, n] = R[m, n] + (b2[n] + sum_i sum_{j<f} Y[m, i f + j] W2[i f + j, n])
 *   Y device bf16 [M, F]; R device bf16 [M, H]; Z device [M, H] (bf16, or fp32 with
 *   TPMLP_FLAG_Z_FP32). Z may be R itself. M == 0 is a no-op.
 * Errors: INVALID_ARG, NOT_PACKED, MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_gemm2_residual(tpmlp_ctx *ctx, const void *Y, int64_t M, void *Z,
                                   const void *R, void *stream);

/*
 * Training forward pass of the block: tpmlp_forward, and the activations the backward pass
 * needs are kept in the caller's buffers.
 *   Ysave  device bf16 [B*S, F]: Y = GeLU(X W1 + b1) (the first GEMM's output); in a
 *          TPMLP_FLAG_SWIGLU context Y = SiLU(G) * U
 *   Asave  device bf16 [B*S, F]: the pre-activation A = X W1 + b1; in a TPMLP_FLAG_SWIGLU
 *          context [B*S, 2F]: G = X Wg + bg in columns [0, F) and U = X Wu + bu in [F, 2F)
 * Errors: as tpmlp_forward.
 */
TPMLP_API int tpmlp_forward_train(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S, void *Z,
                                  void *Ysave, void *Asave, void *stream);

/*
 * Backward pass of the block. The pages repeat the split for the gradients, with one more
 * All-Reduce per block (分布式训练系列第四篇 §4.2-4.3; AI大模型分布式训练 §2.4); here that sum
 * over shards is again taken in the fp32 accumulator:
 *   dA  = (dZ W2^T) * GeLU'(A)     per column shard, GeLU'(a) = Phi(a) + a phi(a)
 *   dX  = sum_i dA_i W1_i^T        the backward All-Reduce, in the accumulator
 *   dW1 = X^T dA,  db1 = sum over tokens of dA
 *   dW2 = Y^T dZ,  db2 = sum over tokens of dZ
 * Inputs (device): dZ bf16 [B*S, H]; X bf16 [B*S, H]; Ysave, Asave from tpmlp_forward_train;
 * W1 bf16 [H, F] and W2 bf16 [F, H]: the same weights that were packed, in the caller's own
 * [in, out] layout (read directly; training keeps its parameters). Outputs (device, written,
 * not accumulated): dX [B*S, H] (bf16, or fp32 with TPMLP_FLAG_Z_FP32); dW1 fp32 [H, F];
 * db1 fp32 [F]; dW2 fp32 [F, H]; db2 fp32 [H]. The context's Y buffer holds dA meanwhile.
 * Eight launches; deterministic. GeLU blocks only. Errors: as tpmlp_forward.
 */
TPMLP_API int tpmlp_backward(tpmlp_ctx *ctx, const void *dZ, const void *X, const void *Ysave,
                             const void *Asave, const void *W1, const void *W2, int64_t B,
                             int64_t S, void *dX, void *dW1, void *db1, void *dW2, void *db2,
                             void *stream);

/*
 * Backward pass of the gated (TPMLP_FLAG_SWIGLU) block, Z = sum_i (SiLU(G_i) * U_i) W2_i + b2
 * with G = X Wg + bg and U = X Wu + bu. gate_up_proj is column-parallel and down_proj
 * row-parallel (大模型分布式优化技术（一） §5.1; AI大模型分布式训练 §6.1), and the backward pass
 * repeats the split with one more sum over shards (分布式训练系列第四篇 §4.2-4.3). By the chain rule:
 *   dY  = dZ W2^T                      per column shard
 *   dU  = dY * SiLU(G),   dG = dY * U * SiLU'(G),   SiLU'(g) = s (1 + g (1 - s)), s = sigma(g)
 *   dX  = sum_i (dG_i Wg_i^T + dU_i Wu_i^T)   the backward All-Reduce, in one accumulator
 *                                             (the k gate shards, then the k up shards)
 *   dWg = X^T dG,  dbg = sum over tokens of dG;  dWu = X^T dU,  dbu = sum over tokens of dU
 *   dW2 = Y^T dZ,  db2 = sum over tokens of dZ
 * Inputs (device): dZ bf16 [B*S, H]; X bf16 [B*S, H]; Ysave [B*S, F] and Asave [B*S, 2F]
 * from tpmlp_forward_train on this context; Wg, Wu bf16 [H, F] and W2 bf16 [F, H]: the
 * weights that were packed, in the caller's [in, out] layout. Outputs (device, written, not
 * accumulated): dX [B*S, H] (bf16, or fp32 with TPMLP_FLAG_Z_FP32); dWg, dWu fp32 [H, F];
 * dbg, dbu fp32 [F]; dW2 fp32 [F, H]; db2 fp32 [H]. dG and dU go to a context buffer of
 * [B*S, 2F] bf16, allocated on first use and grown when B*S grows (that growth
 * synchronises the device). Eleven launches; deterministic.
 * Errors: INVALID_ARG (also for a context without TPMLP_FLAG_SWIGLU), NOT_PACKED,
 * MISALIGNED, UNSUPPORTED_SHAPE, OOM, CUDA.
 */
TPMLP_API int tpmlp_backward_swiglu(tpmlp_ctx *ctx, const void *dZ, const void *X,
                                    const void *Ysave, const void *Asave, const void *Wg,
                                    const void *Wu, const void *W2, int64_t B, int64_t S,
                                    void *dX, void *dWg, void *dbg, void *dWu, void *dbu,
                                    void *dW2, void *db2, void *stream);

/*
 * Read and clear the device status word that the kernels set when a bounded wait gives up
 * (synchronises `stream`). Returns TPMLP_OK, TPMLP_ERR_DEVICE_TIMEOUT or TPMLP_ERR_CUDA.
 * *detail (optional) receives the raw word: which barrier wait gave up.
 */
TPMLP_API int tpmlp_get_status(tpmlp_ctx *ctx, void *stream, int32_t *detail);

/*
 * Where the packed weights live (for tests that unpack and compare them bit for bit).
 *   which: 0 = W1p bf16 [k][f][H], 1 = W2p bf16 [k][H][f], 2 = b1 fp32 [F], 3 = b2 fp32 [H];
 *   for a TPMLP_FLAG_SWIGLU context W1p is [k][2f][H] and b1 [2F], gate/up interleaved in
 *   blocks of G rows (see tpmlp_pack_shards_swiglu). When H is a multiple of 256 and
 *   TPMLP_FLAG_SINGLE_SM is not set (the second GEMM runs on CTA pairs), W2p is stored in
 *   contiguous blocks of 128 rows x 64 columns instead: [k][H/128][f/64][128][64], i.e.
 *   W2p[i][n][j] sits at ((i (H/128) + n/128) (f/64) + j/64) 8192 + (n%128) 64 + j%64.
 * *ptr receives a device pointer owned by the context; *bytes its size.
 * Errors: INVALID_ARG, NOT_PACKED.
 */
TPMLP_API int tpmlp_packed_buffer(const tpmlp_ctx *ctx, int32_t which, const void **ptr, int64_t *bytes);

/*
 * Forward pass that allocates nothing (no counterpart on the pages; an addition for
 * callers that cannot call cudaMalloc when they run the block -- e.g. a serving process
 * whose own allocator has taken the device's free memory at start-up, or a latency-critical
 * stream on which an allocation's implicit device synchronisation is not acceptable).
 *
 * Same arguments, result and errors as tpmlp_forward, but the intermediate activations
 * Y [B*S, F] (bf16) are written to a fixed array compiled into the library,
 * TPMLP_NOALLOC_SCRATCH_BYTES long, instead of the context's buffer. This call makes no
 * cudaMalloc/cudaFree and no other allocating call. Every GPU that loads the library holds
 * that array until the process exits.
 *  - B*S*F*2 > TPMLP_NOALLOC_SCRATCH_BYTES is rejected with TPMLP_ERR_UNSUPPORTED_SHAPE
 *    (tpmlp_last_error states the sizes); nothing is launched.
 *  - The context's device must be current, as for every call (checked on every call).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *    and caches it with the id of the CUDA context it was found in; make that first call
 *    before any stream capture. After cudaDeviceReset the device's next context has another
 *    id, and the next call looks the address up again (contexts created before the reset are
 *    invalid anyway and must be destroyed).
 *  - All calls in the process share the one array per device, and it keeps the previous
 *    call's contents (nothing in it needs to start at zero). Calls whose kernels overlap on
 *    the GPU -- on different streams, or from different contexts -- race on it; serialise them.
 * The weights still come from a context created and packed beforehand.
 */
#define TPMLP_NOALLOC_SCRATCH_BYTES (32ll << 20) /* 32 MiB */
TPMLP_API int tpmlp_forward_noalloc(tpmlp_ctx *ctx, const void *X, int64_t B, int64_t S, void *Z,
                                    void *stream);

/*
 * The two parallel linear layers on their own, all k shards on this GPU: the projections of
 * the pages' tensor-parallel attention (AI大模型分布式训练 §2.3: Q/K/V is a ColumnParallelLinear
 * with the heads split into k groups, the output projection a RowParallelLinear followed by
 * the All-Reduce). W is [K, N] in math orientation (out = X W + b), b is [N].
 *   TPMLP_LINEAR_COLUMN  W split by columns: out[:, i f:(i+1) f] = X W_i + b_i, f = N / k
 *                        (the outputs of the shards side by side; the first GEMM's kernel
 *                        with a bias-only epilogue)
 *   TPMLP_LINEAR_ROW     W split by rows, X by the matching columns (f = K / k):
 *                        out = sum_i X_i W_i + b, the sum over shards taken in the second
 *                        GEMM's fp32 accumulator (the All-Reduce on chip), b added once
 * Shapes: K, N multiples of 64; the sharded dimension divisible by k into multiples of 64.
 * flags: 0, TPMLP_FLAG_Z_FP32 (fp32 output), TPMLP_FLAG_SINGLE_SM, TPMLP_FLAG_FIXED_ORDER.
 * The context is used with tpmlp_linear_pack / tpmlp_linear_forward / tpmlp_destroy (and the
 * diagnostic calls); the MLP-block entry points reject it with TPMLP_ERR_INVALID_ARG.
 * Errors: INVALID_ARG, UNSUPPORTED_SHAPE, ARCH, OOM, CUDA.
 */
#define TPMLP_LINEAR_COLUMN 0
#define TPMLP_LINEAR_ROW 1
TPMLP_API int tpmlp_linear_create(tpmlp_ctx **out, int32_t kind, int64_t K, int64_t N, int32_t k,
                                  uint32_t flags);

/*
 * Pack a linear layer's weight: W device bf16 [K, N], b device bf16 [N] (may be freed once the
 * stream has passed this call). Errors: INVALID_ARG (not a linear context), MISALIGNED, CUDA.
 */
TPMLP_API int tpmlp_linear_pack(tpmlp_ctx *ctx, const void *W, const void *b, void *stream);

/*
 * out = the layer applied to X: X device bf16 [M, K]; out device [M, N] (bf16, or fp32 with
 * TPMLP_FLAG_Z_FP32). One kernel launch; M == 0 is a no-op.
 * Errors: INVALID_ARG, NOT_PACKED, MISALIGNED, UNSUPPORTED_SHAPE, CUDA.
 */
TPMLP_API int tpmlp_linear_forward(tpmlp_ctx *ctx, const void *X, int64_t M, void *out,
                                   void *stream);

/* Release everything the context owns (synchronises its device first). NULL is a no-op. */
TPMLP_API void tpmlp_destroy(tpmlp_ctx *ctx);

/* Static, human-readable text for a tpmlp_status value. */
TPMLP_API const char *tpmlp_strerror(int status);

/* The last CUDA error text recorded on this context ("" if none); valid until the next call. */
TPMLP_API const char *tpmlp_last_error(const tpmlp_ctx *ctx);

/* The number of kernel launches this context has issued so far (pack + forward). */
TPMLP_API int64_t tpmlp_launch_count(const tpmlp_ctx *ctx);

/*
 * The rates two host-side planners work from (no counterpart on the pages; they shape the
 * schedule, never the result):
 *   gemm_flops  dense bf16 FLOP/s the GEMMs sustain on the whole device; sets the time of a
 *               round of output tiles, which the split rule of the CTA-pair kernel (spread the
 *               last, partial wave's reductions over all pairs?) and the row-chunk planner of
 *               tpmlp_forward_host weigh against the two rates below
 *   dram_Bps    HBM bytes/s a stream of reads reaches (the split rule's cost of re-reading a
 *               split tail's operands)
 *   copy_Bps    page-locked host <-> device bytes/s per direction with copies both ways at
 *               once (tpmlp_forward_host's chunk sizes)
 * tpmlp_create derives them from the device: SMs x 8192 FLOP per clock x the maximum SM clock
 * x 0.67 (the share a bf16 GEMM holds under a GB300's power cap); 2 x memory clock x bus
 * width x 0.8; and 168 GB/s (measured over NVLink-C2C). A caller that has measured its own
 * may set them; 0 keeps a rate as it is. Results never depend on them: only which tiles are
 * split (and so, by TPMLP_FLAG_FIXED_ORDER's rule, the last bits of split tiles) and the
 * host-buffer chunk sizes do.
 * Errors: INVALID_ARG (NULL context or pointer, a negative, NaN or absurd (> 1e18) rate).
 */
TPMLP_API int tpmlp_set_device_rates(tpmlp_ctx *ctx, double gemm_flops, double dram_Bps,
                                     double copy_Bps);
TPMLP_API int tpmlp_get_device_rates(const tpmlp_ctx *ctx, double *gemm_flops, double *dram_Bps,
                                     double *copy_Bps);

/*
 * An id of the library build: 16 hex digits of SHA-256 over its CUDA/C++ sources and compile
 * flags (no counterpart on the pages). Measurements recorded against one build of the kernels
 * (DRAM traffic from a profiler, say) can be checked against the build that is running.
 * Static string.
 */
TPMLP_API const char *tpmlp_build_id(void);

#ifdef __cplusplus
}
#endif

#endif /* TPMLP_H */
