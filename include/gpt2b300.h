/*
 * gpt2b300.h -- C ABI of libgpt2b300.so: one GPT-2 training step (forward
 * with loss, zero_grad, backward, AdamW update) on one NVIDIA B300 (sm_103a).
 *
 * The calls follow the decomposition of llm.c's train_gpt2.c as described on
 * the page «llm.c：Andrej Karpathy带你从零复现LLM», section
 * «核心代码解读：train_gpt2.c»: item 2 (GPT2Config, ParameterTensors,
 * ActivationTensors, the GPT2 struct) and item 3 (build, gpt2_forward,
 * gpt2_zero_grad, gpt2_backward, gpt2_update with AdamW).  The single
 * preallocated buffer that every weight and activation points into is the
 * design of page «千行C代码训完GPT-2», section «纯CUDA也可训».
 *
 * Conventions shared by every call:
 *  - Every function returns a status code (GPT2_OK = 0, negative = error,
 *    positive = warning) unless stated otherwise; gpt2_status_string() names it.
 *  - A handle orders all of its device work on the CUDA stream given to
 *    gpt2_build().  Inside a backward pass some gradient work runs on two
 *    streams the handle owns; they fork from that stream and are joined back
 *    into it before the call returns, so to the caller every call is ordered
 *    on the given stream.  Calls on one handle must not run concurrently (the
 *    handle is not thread-safe); different handles are independent.
 *  - Host pointers are read or written during the call only and never kept.
 *  - After GPT2_ERR_DEVICE_TIMEOUT or GPT2_ERR_CUDA the handle is poisoned:
 *    every later call except gpt2_free() returns the same error.
 *  - Flat parameter layout (elements, fp32), each per-layer tensor stacked
 *    over L: wte (Vp,C), wpe (maxT,C), ln1w (L,C), ln1b (L,C),
 *    qkvw (L,3C,C), qkvb (L,3C), attprojw (L,C,C), attprojb (L,C),
 *    ln2w (L,C), ln2b (L,C), fcw (L,4C,C), fcb (L,4C), fcprojw (L,C,4C),
 *    fcprojb (L,C), lnfw (C), lnfb (C).  Linear weights are (out, in)
 *    row-major: y = x W^T + b.  wte rows [V, Vp) are padding and stay 0.
 *    Gradients and the AdamW moments m, v use the same layout.
 */
#ifndef GPT2B300_H
#define GPT2B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define GPT2_OK 0
#define GPT2_ERR_ARG (-1)            /* NULL handle/pointer, t < 1, bad config */
#define GPT2_ERR_SHAPE (-2)          /* B > maxB, T > maxT, T > max_seq_len, B or T < 1 */
#define GPT2_ERR_TOKEN_RANGE (-3)    /* a token id outside [0, vocab_size) */
#define GPT2_ERR_STATE (-4)          /* backward without a forward that had targets */
#define GPT2_ERR_ARENA (-5)          /* caller arena too small or not 256-byte aligned */
#define GPT2_ERR_CUDA (-6)           /* a CUDA runtime/driver error; handle poisoned */
#define GPT2_ERR_DEVICE_TIMEOUT (-7) /* a bounded device-side wait expired; handle poisoned */
#define GPT2_WARN_NONFINITE 1        /* the loss is NaN or Inf; it is still returned */

/* gemm_precision values. */
#define GPT2_PREC_FP32 0 /* fp32 operands (3xTF32 split products), fp32 everything */
#define GPT2_PREC_BF16 1 /* bf16 matmul/attention operands, fp32 accumulate, fp32 master/AdamW */

/* GPT2Config (item 2 of the page above) plus the padded vocabulary, the
 * matmul operand precision and the architecture variant.  Requirements:
 * channels % num_heads == 0, channels % 64 == 0, head size
 * (channels/num_heads) in {16, 32, 64, 128}, vocab_size <= padded_vocab_size,
 * padded_vocab_size % 64 == 0, llama in {0, 1}.
 * llama = 1 selects the Llama-style variant that the page «千行C代码训完GPT-2»
 * (新智元) names as llm.c's next architectures (RMSNorm in place of layernorm,
 * new layers such as RoPE): every layernorm becomes RMSNorm (y = x rstd w,
 * rstd = 1/sqrt(mean(x^2) + 1e-5), no shift), q and k get rotary position
 * embeddings after the QKV matmul (pair (2i, 2i+1) of each head turned by
 * t * 10000^(-2i/hs) radians), there is no learned position table and no
 * linear bias.  Those tensors keep their places in the flat parameter layout
 * with zero elements, so the layout is GPT-2's minus wpe, every bias and every
 * layernorm shift. */
typedef struct {
  int max_seq_len;
  int vocab_size;
  int padded_vocab_size;
  int num_layers;
  int num_heads;
  int channels;
  int gemm_precision;
  int llama;
} gpt2_config;

typedef struct gpt2_t gpt2_t;

/* Device bytes one handle needs for batches up to (maxB, maxT): parameters,
 * gradients, AdamW m and v, activations, activation gradients and scratch.
 * Returns 0 for an invalid config or shape (maxT > max_seq_len, or more than
 * 4,194,304 tokens maxB * maxT). */
size_t gpt2_arena_bytes(const gpt2_config* cfg, int maxB, int maxT);

/* Creates a handle and initialises the parameters from `seed`: matrices
 * N(0, 0.02) (attprojw, fcprojw additionally x 1/sqrt(2L)), biases 0,
 * layernorm gains 1, shifts 0, padded wte rows 0, drawn with SplitMix64 +
 * Box-Muller so that flat element i uses normal number i of the stream.
 * AdamW moments start at 0.
 *  dev_arena   : NULL -> the library allocates (and frees) the arena;
 *                otherwise a device buffer of >= gpt2_arena_bytes() bytes,
 *                256-byte aligned, owned by the caller and kept alive until
 *                gpt2_free().
 *  cuda_stream : a cudaStream_t, or NULL for the legacy default stream.
 * The call synchronises the stream once before returning. */
int gpt2_build(gpt2_t** out, const gpt2_config* cfg, uint64_t seed, int maxB, int maxT, void* dev_arena,
               size_t arena_bytes, void* cuda_stream);

/* gpt2_forward (item 3): token embedding, L transformer blocks, final
 * layernorm, tied LM head, and -- when targets != NULL -- the softmax
 * cross-entropy over the vocab_size real columns with the loss gradient
 * dlogits = (softmax - onehot)/(B*T) computed in the same pass.
 *  inputs, targets : host int32 arrays of B*T token ids (row-major (B,T));
 *                    targets may be NULL (logits only; backward then fails
 *                    with GPT2_ERR_STATE).
 *  loss_out        : host float, or NULL.  When non-NULL the call
 *                    synchronises the stream and stores the mean loss over
 *                    the B*T positions (-1.0f when targets is NULL); it
 *                    returns GPT2_WARN_NONFINITE for a NaN/Inf loss.  When
 *                    NULL the call returns once the work is enqueued.
 * Token ids are validated on the host before any work is enqueued. */
int gpt2_forward(gpt2_t* m, const int32_t* inputs, const int32_t* targets, int B, int T, float* loss_out);

/* Same as gpt2_forward with device-resident token arrays (B*T int32 each,
 * targets may be NULL).  Never synchronises.  An out-of-range id is detected
 * on the device: the step's results are then undefined and the next
 * gpt2_sync() returns GPT2_ERR_TOKEN_RANGE. */
int gpt2_forward_device(gpt2_t* m, const int32_t* d_inputs, const int32_t* d_targets, int B, int T);

/* Text generation: the page «llm.c：Andrej Karpathy带你从零复现LLM», section
 * «核心代码解读：train_gpt2.c», item 5 (sample_mult draws an index from a
 * probability distribution; the main loop generates a sequence with it).
 * For t = n_prompt .. n_total-1: one forward without targets over batch row
 * 0 and all n_total positions (positions not yet generated hold tokens[0];
 * causal attention keeps them out of the row that is read), then
 * tokens[t] = the first index i < vocab_size whose cumulative softmax
 * probability of logits row t-1 exceeds coins[t - n_prompt] (inverse-CDF
 * sampling; the last index with nonzero weight if rounding leaves the coin
 * above every prefix).
 *  tokens  : host int32[n_total]; in: the prompt in [0, n_prompt), ids in
 *            [0, vocab_size); out: prompt followed by the generated ids.
 *  coins   : host float[n_total - n_prompt], each in [0, 1), e.g. uniform
 *            draws of the caller's generator (the library draws none).
 *  1 <= n_prompt < n_total <= min(maxT, max_seq_len); the handle needs maxB >= 1.
 * Synchronises the stream.  Returns GPT2_ERR_ARG for a bad count or a coin
 * outside [0, 1), GPT2_ERR_TOKEN_RANGE for a bad prompt id, GPT2_ERR_SHAPE when
 * n_total does not fit the handle.  Overwrites the logits, so a following
 * gpt2_backward() fails with GPT2_ERR_STATE. */
int gpt2_sample(gpt2_t* m, int32_t* tokens, int n_prompt, int n_total, const float* coins);

/* Synchronises the handle's stream; reports device-side errors recorded since
 * the previous sync and, when loss_out != NULL, stores the last mean loss. */
int gpt2_sync(gpt2_t* m, float* loss_out);

/* gpt2_zero_grad (item 3): sets every parameter gradient to 0.  Activation
 * gradients are overwritten by gpt2_backward and need no clearing. */
int gpt2_zero_grad(gpt2_t* m);

/* gpt2_backward (item 3): ACCUMULATES (+=) the gradient of the mean loss of
 * the last forward into the parameter gradients.  GPT2_ERR_STATE if the last
 * forward had no targets.  Does not synchronise. */
int gpt2_backward(gpt2_t* m);

/* gpt2_update (item 3): one AdamW step over every parameter, step number
 * t >= 1 (bias corrections 1 - beta^t), decoupled weight decay:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr * ((m/(1-b1^t)) / (sqrt(v/(1-b2^t)) + eps) + weight_decay * p).
 * Does not synchronise. */
int gpt2_update(gpt2_t* m, float lr, float beta1, float beta2, float eps, float weight_decay, int t);

/* One whole step -- forward (device tokens), zero_grad, backward, update --
 * enqueued as a single unit; with use_graph != 0 the sequence is captured
 * once per (B, T) into a CUDA graph and replayed.  Never synchronises. */
int gpt2_train_step_device(gpt2_t* m, const int32_t* d_inputs, const int32_t* d_targets, int B, int T, float lr,
                           float beta1, float beta2, float eps, float weight_decay, int t, int use_graph);

/* One whole step from HOST token arrays, the call a training loop makes:
 * copies the B*T inputs and targets to the device (pinned host memory makes
 * the copies asynchronous), validates them on the host, replays the
 * captured step (forward with loss, zero_grad, backward, AdamW step t) and
 * synchronises to store the step's mean loss in *loss_out (non-NULL).
 * Returns GPT2_WARN_NONFINITE for a NaN/Inf loss. */
int gpt2_train_step(gpt2_t* m, const int32_t* inputs, const int32_t* targets, int B, int T, float lr, float beta1,
                    float beta2, float eps, float weight_decay, int t, float* loss_out);

/* Kernel timer for roofline measurement.  kind selects one kernel class
 * (0 off, 1 matmuls, 2 AdamW, 3 fused cross-entropy, 4 attention forward,
 * 5 attention backward, 6 layernorm, 7 embedding forward); while it is on, every
 * launch of that class is bracketed by CUDA events on the handle's stream
 * and steps run without graph replay.  gpt2_kernel_timer() resets the
 * totals; gpt2_kernel_timer_read() synchronises and returns the summed
 * event time (ms), the number of launches and their summed algorithmic work
 * (FLOPs for matmuls, bytes for the others). */
int gpt2_kernel_timer(gpt2_t* m, int kind);
int gpt2_kernel_timer_read(gpt2_t* m, double* total_ms, long long* launches, double* total_work);

/* Test and diagnosis knob for the bounded device-side waits.  Every
 * tensor-core kernel waits on its pipeline barriers for at most this long
 * (wall time) before it records a timeout, lets its copies and MMAs in
 * flight land, frees its tensor memory and returns; the next synchronising
 * call then reports GPT2_ERR_DEVICE_TIMEOUT and poisons the handle (the
 * per-layer gpt2op_* calls return it directly).  Default 1 s; ns = 0
 * restores it.  A limit below 1000 ns makes every such wait give up at its
 * first call -- tests use that to drive the timeout path, the same way every
 * time and without a fault.  Applies to the current device and to every
 * handle and call on it; synchronises the device. */
int gpt2_set_wait_limit_ns(unsigned long long ns);

/* The tile plan of the bf16 tensor-core matmul for an M x N x K product
 * (out[M][N] = sum over K), as the model's steps and gpt2op_matmul_* take it
 * on a GPU with num_sms SMs (148 on a B300).  A host-side query: no device,
 * handle or memory is touched.  *BN receives the output tile width (128, 192
 * or 256; tiles are 128 rows high), *splits the number of K ranges reduced
 * through the split-K workspace (1: none).  no_split != 0: an epilogue that
 * takes column sums (bias gradients), which a K split would bypass.
 * logits != 0: the LM head's epilogue with per-half-tile row statistics (no
 * K split, no 192-wide tiles).  Returns GPT2_ERR_ARG for a non-positive size
 * or SM count or a NULL output.  The pages have no counterpart: it exposes
 * the library's own wave and K-tile cost model for inspection and tests. */
int gpt2_plan_bf16_matmul(int M, int N, int K, int no_split, int logits, int num_sms, int* BN, int* splits);

/* Frees the handle (and the arena if the library allocated it). */
int gpt2_free(gpt2_t* m);

/* Number of elements of the flat (padded) parameter buffer; -1 for NULL. */
long long gpt2_num_parameters(const gpt2_t* m);

/* Host <-> device copies of the flat buffers (n = gpt2_num_parameters());
 * each synchronises the stream.  Used for parity tests and checkpoints. */
int gpt2_get_params(gpt2_t* m, float* host, long long n);
int gpt2_set_params(gpt2_t* m, const float* host, long long n);
int gpt2_get_grads(gpt2_t* m, float* host, long long n);
int gpt2_get_opt_state(gpt2_t* m, float* host_m, float* host_v, long long n);
int gpt2_set_opt_state(gpt2_t* m, const float* host_m, const float* host_v, long long n);

/* Logits of the last forward, (B, T, Vp) fp32, n = B*T*Vp elements.  With
 * GPT2_PREC_BF16 and targets, the forward keeps its logits in bf16 (the
 * cross-entropy reads them once, with row statistics the LM-head matmul
 * computed from the fp32 accumulators); they come back widened to fp32. */
int gpt2_get_logits(gpt2_t* m, float* host, long long n);

/* Number of kernels the last gpt2_forward/backward/update/train_step call
 * enqueued (for launch accounting). */
long long gpt2_last_launch_count(const gpt2_t* m);

/* ---- kernel-level entry points (device buffers, row-major fp32) ----------
 * The per-layer matmul of the page's item 1 (matmul_forward /
 * matmul_backward), run by the same tensor-core kernels the model uses; for
 * per-layer parity tests.  x (N, IC), W (OC, IC), bias (OC), out (N, OC).
 * precision is GPT2_PREC_FP32 (3xTF32 products) or GPT2_PREC_BF16 (the
 * operands are rounded to bf16 into the workspace first, then multiplied by
 * the bf16 kernel with fp32 accumulation).  workspace: a device buffer of
 * gpt2op_matmul_workspace_bytes(N, IC, OC) bytes (scratch; contents not
 * kept).  stream: cudaStream_t or NULL.  Both calls synchronise the stream.
 * IC and OC must be multiples of 4 (fp32) or 8 (bf16): 16-byte rows for TMA;
 * otherwise GPT2_ERR_SHAPE. */
size_t gpt2op_matmul_workspace_bytes(int N, int IC, int OC);
/* out = x W^T (+ bias when bias != NULL). */
int gpt2op_matmul_forward(float* out, const float* x, const float* W, const float* bias, int N, int IC, int OC,
                          int precision, void* workspace, void* stream);
/* dx = dy W (overwritten); dW += dy^T x; dbias += column sums of dy (dbias
 * may be NULL).  dy (N, OC). */
int gpt2op_matmul_backward(float* dx, float* dW, float* dbias, const float* dy, const float* x, const float* W,
                           int N, int IC, int OC, int precision, void* workspace, void* stream);

/* The per-layer causal attention forward of the page's item 1
 * (attention_forward), run by the kernels the model uses; for per-layer
 * parity tests.  qkv (B, T, 3C) row-major: q = columns [0, C), k = [C, 2C),
 * v = [2C, 3C), head h = columns h*hs .. h*hs+hs-1 of each block, hs = C/NH.
 * Writes y (B, T, C) = softmax(q k^T / sqrt(hs), keys t2 <= t) v and
 * lse (B, NH, T), the log-sum-exp of each row of scaled scores.
 * precision GPT2_PREC_FP32: CUDA-core kernel in fp32.  GPT2_PREC_BF16: qkv is
 * rounded to bf16 in the workspace; with hs = 64 and T % 128 == 0 the
 * tensor-core kernel computes the products (softmax in fp32, P rounded to
 * bf16 for P V), otherwise the CUDA-core kernel with bf16-rounded operands.
 * workspace: gpt2op_attention_workspace_bytes(B, T, C) device bytes.
 * Requirements: C % NH == 0, hs <= 128, C % 8 == 0 (else GPT2_ERR_SHAPE).
 * Synchronises the stream. */
size_t gpt2op_attention_workspace_bytes(int B, int T, int C);
int gpt2op_attention_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int NH, int precision,
                             void* workspace, void* stream);

/* The per-layer causal attention backward of the page's item 1
 * (attention_backward): dqkv (B, T, 3C) = the gradient of the loss through
 * y = attention(qkv) for the upstream gradient dy (B, T, C), in the layout of
 * qkv.  The call first runs the attention forward (for y and the row
 * log-sum-exp), then D = rowsum(dy o y), P recomputed from the log-sum-exp,
 * dS = P o (dy v^T - D), dq = dS k / sqrt(hs), dk = dS^T q / sqrt(hs),
 * dv = P^T dy.  precision and requirements as gpt2op_attention_forward (bf16:
 * qkv and dy rounded to bf16; with hs = 64 and T % 128 == 0 the tensor-core
 * kernels: persistent CTAs, one per SM, walk the output row tiles, each tile
 * written by one CTA, no atomics).  dqkv is overwritten.
 * workspace: gpt2op_attention_backward_workspace_bytes(B, T, C, NH) device
 * bytes.  Synchronises the stream. */
size_t gpt2op_attention_backward_workspace_bytes(int B, int T, int C, int NH);
int gpt2op_attention_backward(float* dqkv, const float* dy, const float* qkv, int B, int T, int C, int NH,
                              int precision, void* workspace, void* stream);

/* gpt2op_matmul_backward without a workspace argument: the same products
 * (dx = dy W; dW += dy^T x; dbias += column sums of dy, dbias may be NULL)
 * with the same arguments minus `workspace`.  The pages have no counterpart:
 * this entry point exists for callers that cannot allocate device memory --
 * for example a plugin inside a host application whose allocator already
 * owns the device's memory, or a loop that must not call cudaMalloc because
 * it can synchronise the device.  It allocates nothing and calls no
 * allocating routine.
 * Scratch: one fixed array of 8 MiB + 1280 bytes in the library's device
 * memory, which every GPU that loads the library holds until the process
 * exits.  The first call on a device looks up that array's device address
 * (cudaGetSymbolAddress, with the device current) and caches it; make that
 * first call before any stream capture.  Every call on a device shares the
 * array, and each call clears the part that must start at zero: calls that
 * overlap on the GPU (different streams, or different host threads on one
 * device) race and give wrong results.
 * Limit: with dbias != NULL, ceil(N/64) * OC must be <= 2,097,152 (for
 * example N = 16384 with OC <= 8192): the column-sum partials of the bias
 * gradient fill the array; larger shapes return GPT2_ERR_SHAPE before any
 * device work.  precision must be GPT2_PREC_FP32 (bf16 operand copies would
 * need scratch that grows with the inputs): GPT2_ERR_ARG otherwise.  The fp32
 * products reduce their K splits on chip and use no other scratch.
 * Synchronises the stream. */
int gpt2op_matmul_backward_noalloc(float* dx, float* dW, float* dbias, const float* dy, const float* x,
                                   const float* W, int N, int IC, int OC, int precision, void* stream);

/* Static description of a status code (never NULL). */
const char* gpt2_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GPT2B300_H */
