// gpt2.cu -- the GPT-2 training-step runtime behind the C ABI of
// include/gpt2b300.h: arena planning and carving, the forward / backward /
// AdamW kernel sequences on the handle's stream, CUDA-graph replay of whole
// steps, status codes and host-side validation.
//
// Structure follows llm.c's train_gpt2.c as described on the page
// «llm.c：Andrej Karpathy带你从零复现LLM», section «核心代码解读：train_gpt2.c»
// (items 1-3: layer functions, model structs, build/forward/zero_grad/
// backward/update) and the single preallocated buffer of page
// «千行C代码训完GPT-2», section «纯CUDA也可训».  Unlike the CPU design, the
// activation arena never stores the (T,T) attention matrices: the attention
// kernels keep only the per-row log-sum-exp and recompute probabilities in
// the backward pass.
#include <vector>
#include <math.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <utility>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/gpt2b300.h"
#include "common.cuh"
#include "k_attention_simt.cuh"
#include "k_attention_small.cuh"
#include "k_attention_tc.cuh"
#include "k_attention_tf32.cuh"
#include "k_gemm_bf16.cuh"
#include "k_gemm_tc.cuh"
#include "k_layernorm.cuh"
#include "k_misc.cuh"
#include "k_rope.cuh"
#include "k_sample.cuh"
#include "k_xent.cuh"

#define EXPORT extern "C" __attribute__((visibility("default")))

// split-K workspace (fp32 partial tiles), 32 MB
#define SPLITK_WS_FLOATS ((long long)8 << 20)
// events of the backward's side stream (two per side launch, ~50 launches per backward)
#define SIDE_EVENTS 256
// split-K arrival counters: K is split only when there are fewer than 148 tiles
#define TILE_CTRS 256
// op workspaces start with [error word, 256 B][tile counters, 1 KB]
#define OP_HDR_BYTES 1280
// smallest row chunk of the bias-gradient column sums
#define BIAS_MIN_ROWS 32

enum {
  P_WTE, P_WPE, P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_ATTPROJW, P_ATTPROJB,
  P_LN2W, P_LN2B, P_FCW, P_FCB, P_FCPROJW, P_FCPROJB, P_LNFW, P_LNFB, NUM_PARAMS
};

// ---------------------------------------------------------------------------
// arena plan
// ---------------------------------------------------------------------------
struct Plan {
  size_t total;
  size_t params, grads, m, v, params_bf;
  size_t encoded, ln1, ln1_mean, ln1_rstd, qkv, atty, lse, res2, ln2, ln2_mean, ln2_rstd, fch, fchg, res3;
  size_t lnf, lnf_mean, lnf_rstd, logits, dlogits, losses, loss;
  size_t dres, dln, datty, dqkv, dfch, attD, scratch, sorted, tokens, targets, err, hparams, splitk, tilectr;
  size_t sort_tmp, radix_hist;  // the embedding backward's radix sort (more than SORT_BITONIC_MAX tokens)
  size_t runs;                  // where each id's run of sorted positions starts, and the run count
  // the split-K workspace and tile counters of the weight-gradient side stream (bf16 matmuls only)
  size_t splitk_w, tilectr_w;
  // bf16 operand copies (bf16 matmuls only)
  size_t ln1_bf, qkv_bf, atty_bf, ln2_bf, fchg_bf, lnf_bf, dlogits_bf, dres_bf, dfch_bf, dqkv_bf, datty_bf;
  // bf16 logits, their per-block softmax statistics and the targets' fp32
  // logits (forward with targets, bf16 matmuls)
  size_t logits_bf, xstats, tlogit;
  // one byte per wte row: 1 when the batch's tokens touch it (fused step)
  size_t rowmask;
  // Llama-style variant: (cos, sin) per position and pair, and a zero vector
  // standing in for the biases the variant does not have
  size_t rope, zero_bias;
  size_t scratch_floats;
};

static long long param_count(const gpt2_config* c, long long sizes[NUM_PARAMS]) {
  long long L = c->num_layers, C = c->channels;
  long long s[NUM_PARAMS] = {(long long)c->padded_vocab_size * C, (long long)c->max_seq_len * C, L * C, L * C,
                             L * 3 * C * C, L * 3 * C, L * C * C, L * C, L * C, L * C, L * 4 * C * C, L * 4 * C,
                             L * C * 4 * C, L * C, C, C};
  if (c->llama)  // no position table, no biases, no layernorm shifts: the tensors stay, empty
    s[P_WPE] = s[P_LN1B] = s[P_QKVB] = s[P_ATTPROJB] = s[P_LN2B] = s[P_FCB] = s[P_FCPROJB] = s[P_LNFB] = 0;
  long long n = 0;
  for (int i = 0; i < NUM_PARAMS; i++) {
    if (sizes) sizes[i] = s[i];
    n += s[i];
  }
  return n;
}

static int config_ok(const gpt2_config* c) {
  if (!c) return 0;
  if (c->num_layers < 1 || c->channels < 64 || c->num_heads < 1 || c->max_seq_len < 1) return 0;
  if (c->channels % 64 || c->channels % c->num_heads) return 0;
  int hs = c->channels / c->num_heads;
  if (hs != 16 && hs != 32 && hs != 64 && hs != 128) return 0;
  if (c->channels > 32 * 4 * LN_MAXV4_LIMIT) return 0;
  if (c->vocab_size < 1 || c->vocab_size > c->padded_vocab_size || c->padded_vocab_size % 64) return 0;
  if (c->padded_vocab_size > 65536) return 0;
  if (c->gemm_precision != GPT2_PREC_FP32 && c->gemm_precision != GPT2_PREC_BF16) return 0;
  if (c->llama != 0 && c->llama != 1) return 0;
  return 1;
}

// Tokens per batch a handle may hold (the embedding backward's radix sort
// scans its chunk table in one CTA; 4M tokens is far beyond any workload).
#define MAX_TOKENS ((long long)1 << 22)

static int shape_ok(const gpt2_config* c, int maxB, int maxT) {
  return maxB >= 1 && maxT >= 1 && maxT <= c->max_seq_len && (long long)maxB * maxT <= MAX_TOKENS;
}

// Softmax-statistics blocks per row of the bf16 logits: one per BN/2 columns
// of the LM-head tiles, at most Vp/64 (BN = 128).
static size_t xstats_pitch(size_t Vp) { return (Vp + 63) / 64; }

static size_t plan_arena(const gpt2_config* c, int maxB, int maxT, Plan* p) {
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t at = off;
    off += (bytes + 255) & ~(size_t)255;
    return at;
  };
  long long np = param_count(c, nullptr);
  size_t L = c->num_layers, C = c->channels, NH = c->num_heads, Vp = c->padded_vocab_size;
  size_t BT = (size_t)maxB * maxT;
  size_t F = sizeof(float);
  p->params = take(np * F);
  p->grads = take(np * F);
  p->m = take(np * F);
  p->v = take(np * F);
  p->params_bf = take(c->gemm_precision == GPT2_PREC_BF16 ? np * 2 : 0);
  p->encoded = take(BT * C * F);
  p->ln1 = take(L * BT * C * F);
  p->ln1_mean = take(L * BT * F);
  p->ln1_rstd = take(L * BT * F);
  p->qkv = take(L * BT * 3 * C * F);
  p->atty = take(L * BT * C * F);
  p->lse = take(L * BT * NH * F);
  p->res2 = take(L * BT * C * F);
  p->ln2 = take(L * BT * C * F);
  p->ln2_mean = take(L * BT * F);
  p->ln2_rstd = take(L * BT * F);
  // the MLP pre-activation: fp32, or bf16 with bf16 matmuls (only gelu' reads it)
  p->fch = take(L * BT * 4 * C * (c->gemm_precision == GPT2_PREC_BF16 ? 2 : F));
  p->fchg = take(L * BT * 4 * C * F);
  p->res3 = take(L * BT * C * F);
  p->lnf = take(BT * C * F);
  p->lnf_mean = take(BT * F);
  p->lnf_rstd = take(BT * F);
  p->logits = take(BT * Vp * F);
  p->dlogits = take(BT * Vp * F);
  p->losses = take(BT * F);
  p->loss = take(F);
  p->dres = take(BT * C * F);
  p->dln = take(BT * C * F);
  p->datty = take(BT * C * F);
  p->dqkv = take(BT * 3 * C * F);
  p->dfch = take(BT * 4 * C * F);
  p->attD = take(2 * BT * NH * F);  // D, or the (-lse log2 e, -D) pairs of the tensor-core path
  // scratch: column-sum partials (<= ceil(BT/BIAS_MIN_ROWS) x 4C) and
  // layernorm partials (<= ceil(BT/LNB_MIN_ROWS) x 3C)
  size_t s1 = ((BT + BIAS_MIN_ROWS - 1) / BIAS_MIN_ROWS) * 4 * C;
  size_t s2 = ((BT + LNB_MIN_ROWS - 1) / LNB_MIN_ROWS) * 3 * C;
  p->scratch_floats = s1 > s2 ? s1 : s2;
  p->scratch = take(p->scratch_floats * F);
  p->sorted = take(BT * sizeof(uint32_t));
  p->sort_tmp = take(BT * sizeof(uint32_t));
  p->radix_hist = take(256 * ((BT + RADIX_CHUNK - 1) / RADIX_CHUNK) * sizeof(int));
  p->runs = take((BT + 1) * sizeof(int));  // the run starts, then their count
  p->tokens = take(BT * sizeof(int));
  p->targets = take(BT * sizeof(int));
  p->err = take(sizeof(int));
  p->hparams = take(16 * F);
  p->splitk = take(SPLITK_WS_FLOATS * F);
  p->tilectr = take(TILE_CTRS * sizeof(int));
  const bool bf16_gemm = c->gemm_precision == GPT2_PREC_BF16;
  p->splitk_w = take(bf16_gemm ? SPLITK_WS_FLOATS * F : 0);
  p->tilectr_w = take(bf16_gemm ? TILE_CTRS * sizeof(int) : 0);
  const size_t H = c->gemm_precision == GPT2_PREC_BF16 ? 2 : 0;  // bytes per bf16 copy element (0: none)
  p->ln1_bf = take(L * BT * C * H);
  p->qkv_bf = take(L * BT * 3 * C * H);
  p->atty_bf = take(L * BT * C * H);
  p->ln2_bf = take(L * BT * C * H);
  p->fchg_bf = take(L * BT * 4 * C * H);
  p->lnf_bf = take(BT * C * H);
  p->dlogits_bf = take(BT * Vp * H);
  p->dres_bf = take(BT * C * H);
  p->dfch_bf = take(BT * 4 * C * H);
  p->dqkv_bf = take(BT * 3 * C * H);
  p->datty_bf = take(BT * C * H);
  p->logits_bf = take(BT * Vp * H);
  p->xstats = take(H ? BT * xstats_pitch(Vp) * sizeof(float2) : 0);
  p->tlogit = take(H ? BT * F : 0);
  p->rowmask = take(Vp);
  const size_t ll = c->llama ? 1 : 0;
  p->rope = take(ll * (size_t)maxT * (C / NH / 2) * 2 * F);
  p->zero_bias = take(ll * 4 * C * F);
  p->total = off;
  return off;
}

// ---------------------------------------------------------------------------
// the handle
// ---------------------------------------------------------------------------
struct gpt2_t {
  gpt2_config cfg;
  int maxB, maxT;
  long long np;
  long long psize[NUM_PARAMS];
  Plan plan;
  char* arena;
  int own_arena;
  cudaStream_t stream;
  float *params, *grads, *m, *v;
  uint16_t* params_bf;
  float* P[NUM_PARAMS];
  float* G[NUM_PARAMS];
  float *encoded, *ln1, *ln1_mean, *ln1_rstd, *qkv, *atty, *lse, *res2, *ln2, *ln2_mean, *ln2_rstd, *fch, *fchg,
      *res3;
  float *lnf, *lnf_mean, *lnf_rstd, *logits, *dlogits, *losses, *loss;
  float *dres, *dln, *datty, *dqkv, *dfch, *attD, *scratch, *splitk, *splitk_w;
  uint32_t *sorted, *sort_tmp;
  int *radix_hist, *runs, *nruns;
  int *tokens, *targets, *err, *tilectr, *tilectr_w;
  uint16_t *ln1_bf, *qkv_bf, *atty_bf, *ln2_bf, *fchg_bf, *lnf_bf, *dlogits_bf, *dres_bf, *dfch_bf, *dqkv_bf,
      *datty_bf;
  uint16_t* logits_bf;  // the LM head's output of a bf16 forward with targets
  float2* xstats;       // its per-block softmax statistics, xstats_pitch(Vp) per row
  float* tlogit;        // the targets' fp32 logits
  int logits_in_bf;     // 1: the last forward's logits are in logits_bf (bf16), 0: in logits (fp32)
  uint8_t* rowmask;     // per wte row: touched by the batch's tokens (fused step)
  float* hparams;
  float2* rope;       // [maxT][hs/2] (cos, sin) of t * 10000^(-2i/hs) (Llama-style variant)
  float* zero_bias;   // 4C zeros: the bias operand of the variant's linear layers
  int B, T, have_targets, fwd_done;
  // 1: the backward adds into the gradients (gpt2_backward); 0: it stores
  // them (the fused training step, whose gradients would otherwise be zeroed
  // first -- every gradient element is written exactly once there)
  int grad_accumulate;
  int poisoned;
  long long launches;
  // graph replay of whole steps
  cudaGraphExec_t gexec;
  int gB, gT;
  long long g_launches;
  int capturing;
  // Side stream for the backward's column-sum finishes (bias, layernorm gain
  // and shift gradients): nothing but AdamW reads their outputs, so they run
  // beside the main stream instead of between two dependent matmuls.  sev is
  // a ring of events; rd_* is the event after which the side stream no
  // longer reads that buffer (-1: no pending reader), side_last the last
  // side event (the join before the update).
  cudaStream_t side;
  cudaEvent_t sev[SIDE_EVENTS];
  int sev_next, side_last, rd_scratch, rd_dfch, rd_dqkv;
  // A second, lower-priority side stream for the per-layer weight-gradient
  // matmuls, beside the input-gradient chain (bf16 matmuls there use their own
  // split-K workspace and tile counters, splitk_w and tilectr_w); wd_* as
  // rd_* for it.
  cudaStream_t side_w;
  int side_w_last, wd_dres, wd_dfch, wd_dqkv;
  // A third side stream, also at the lowest priority, for the AdamW updates of
  // the fused step: layer l's parameters are updated there as soon as the
  // backward has finished their gradients, beside the backward of the layers
  // below (upd_layers: 1 while the fused step enqueues its backward;
  // side_u_last: the event after its last update, -1 for none).
  cudaStream_t side_u;
  int upd_layers, side_u_last;
  // kernel timer: event pairs around every launch of one kernel class
  int timer_kind;
  cudaEvent_t* tev;
  double* twork;
  int tcap, tused;
  double t_ms, t_work;
  long long t_launches;
};

// Kernel classes the timer can bracket.
enum TimerKind { TK_NONE = 0, TK_GEMM = 1, TK_ADAMW = 2, TK_XENT = 3, TK_ATTN_FWD = 4, TK_ATTN_BWD = 5,
                 TK_LAYERNORM = 6, TK_ENCODER = 7 };

static void timer_drain(gpt2_t* m) {
  if (!m->tused) return;
  cudaEventSynchronize(m->tev[2 * m->tused - 1]);
  for (int i = 0; i < m->tused; i++) {
    float ms = 0.f;
    cudaEventElapsedTime(&ms, m->tev[2 * i], m->tev[2 * i + 1]);
    m->t_ms += ms;
    m->t_work += m->twork[i];
    m->t_launches++;
  }
  m->tused = 0;
}

static inline void timer_begin(gpt2_t* m, int kind, double work) {
  if (m->timer_kind != kind || m->capturing || !m->tev) return;
  if (m->tused == m->tcap) timer_drain(m);
  m->twork[m->tused] = work;
  cudaEventRecord(m->tev[2 * m->tused], m->stream);
}

static inline void timer_end(gpt2_t* m, int kind) {
  if (m->timer_kind != kind || m->capturing || !m->tev) return;
  cudaEventRecord(m->tev[2 * m->tused + 1], m->stream);
  m->tused++;
}

#define KCHECK(m)                                  \
  do {                                             \
    cudaError_t e_ = cudaGetLastError();           \
    if (e_ != cudaSuccess) {                       \
      (m)->poisoned = GPT2_ERR_CUDA;               \
      fprintf(stderr, "gpt2b300: %s (%s:%d)\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      return GPT2_ERR_CUDA;                        \
    }                                              \
  } while (0)

#define CCHECK(m, call)                            \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) {                       \
      (m)->poisoned = GPT2_ERR_CUDA;               \
      fprintf(stderr, "gpt2b300: %s (%s:%d)\n", cudaGetErrorString(e_), __FILE__, __LINE__); \
      return GPT2_ERR_CUDA;                        \
    }                                              \
  } while (0)

// Every kernel is launched with programmatic stream serialization: the next
// kernel in the stream may start (its CTAs run their set-up, then wait at
// griddepcontrol.wait inside the kernel) while this one drains.  Kernels call
// griddepcontrol.wait before their first global-memory access, so every
// read-after-write and write-after-read on the stream stays ordered.
static int g_pdl = 1;

template <typename... KArgs, typename... Args>
static void launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 1 : 0;
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);  // errors surface at the next KCHECK
}

static int grid_for(long long n, int threads, int cap = 148 * 16) {
  long long g = (n + threads - 1) / threads;
  if (g > cap) g = cap;
  if (g < 1) g = 1;
  return (int)g;
}

// ---------------------------------------------------------------------------
// matmul launcher
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;

static int get_encoder() {
  if (g_encode_tiled) return 1;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn) {
    cudaGetLastError();
    return 0;
  }
  g_encode_tiled = (PFN_cuTensorMapEncodeTiled_v12000)fn;
  return 1;
}

// Tensor map of an fp32 operand stored as `outer` rows of pitch `ld` elements
// with `inner` valid (contiguous) elements per row.  K-major tiles are
// 32 x 128 boxes with the 128-byte swizzle; MN-major tiles are unswizzled
// 128 x 32 boxes.  Out-of-range elements load as zero.
static int make_operand_map(CUtensorMap* tm, const float* base, int kmajor, long long outer, long long inner,
                            long long ld) {
  if (!get_encoder()) return 0;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
  cuuint32_t box_k[2] = {(cuuint32_t)tc::BK, (cuuint32_t)tc::BM};
  cuuint32_t box_mn[2] = {(cuuint32_t)tc::BM, (cuuint32_t)tc::BK};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void*)base, dims, strides,
                              kmajor ? box_k : box_mn, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              kmajor ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// One matmul acc(i,j) = sum_k A(i,k) B(j,k) with a fused epilogue.  The
// fp32 pointers feed the 3xTF32 kernel, the bf16 ones the bf16 kernel.
struct MatmulDesc {
  int M, N, K;
  const float* A;
  long long lda;
  int a_kmajor;  // 1: A stored (M, lda) with K contiguous; 0: stored (K, lda) with M contiguous
  const float* B;
  long long ldb;
  int b_kmajor;  // 1: B stored (N, ldb) with K contiguous; 0: stored (K, ldb) with N contiguous
  EpiArgs epi;
  const uint16_t* Abf;  // the same operands in bf16 (bf16 matmuls)
  const uint16_t* Bbf;
};

// Clusters of s CTAs of the fp32 matmul (one CTA per SM: its shared memory
// fills the SM) that the GPU holds at once, s = 1..8, and the SM count; filled
// once per process after the kernel's shared-memory limit is set.  A cluster
// sits inside one GPC, so the SMs of a GPC beyond a multiple of s stay idle:
// at s = 3 a 148-SM B300 holds 45 clusters (135 CTAs), not 49.
// Per device: the SM count and the clusters of s CTAs of the fp32 matmul that
// the GPU holds at once (s = 1..8), queried with that device current once its
// kernels' shared-memory limits are set (kernel attributes apply per device);
// attr: 0 not yet set, 1 set, -1 failed.
#define MAX_DEVICES 64
struct DevInfo {
  int num_sms;
  int max_clusters[9];
  int attr;
};
static DevInfo g_dev[MAX_DEVICES];
static std::mutex g_dev_mu;

static int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) {
    cudaGetLastError();
    return -1;
  }
  return dev;
}

// the current device's entry (device 0's when the lookup fails)
static const DevInfo& dev_info() {
  const int d = current_device();
  return g_dev[d < 0 ? 0 : d];
}

static cudaError_t query_cluster_limits(int dev, DevInfo* di) {
  cudaError_t e = cudaDeviceGetAttribute(&di->num_sms, cudaDevAttrMultiProcessorCount, dev);
  di->max_clusters[1] = di->num_sms;
  for (int s = 2; s <= 8 && e == cudaSuccess; s++) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, 1, s);
    cfg.blockDim = dim3(tc::THREADS);
    cfg.dynamicSmemBytes = tc::SMEM_BYTES;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 1;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = s;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, tc::gemm_tf32x3_kernel, &cfg);
    di->max_clusters[s] = n;
  }
  return e;
}

// Split K so that small-M products still fill the SMs.  The splits of a tile
// form one thread-block cluster (at most 8 CTAs, the portable cluster size)
// and are reduced through distributed shared memory in split order.  Cost of
// s splits in units of one K tile of the main loop: waves x (K tiles per
// split + pipeline fill and epilogue) + the cluster reduction, a wave being
// as many clusters as the GPU holds at once.  A tile beyond the first wave
// doubles the time, so s is chosen against the cluster limit above.
static int choose_splits(int M, int N, int K) {
  const DevInfo& di = dev_info();
  const int num_sms = di.num_sms;
  const int* max_clusters = di.max_clusters;
  const long long tiles = (long long)ceil_div(M, tc::BM) * ceil_div(N, tc::BN);
  const int kt = ceil_div(K, tc::BK);
  if (kt < 4) return 1;
  const int FILL = 4, REDUCE = 3;
  int best = 1;
  long long best_cost = ((tiles + num_sms - 1) / num_sms) * (long long)(kt + FILL);
  for (int s = 2; s <= 8 && s <= kt / 2; s++) {
    const int per = ceil_div(kt, s);
    if (ceil_div(kt, per) != s || max_clusters[s] <= 0) continue;  // same split as a smaller s, or no fit
    const long long waves = (tiles + max_clusters[s] - 1) / max_clusters[s];
    const long long cost = waves * (per + FILL) + REDUCE;
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

// Launches the 3xTF32 tensor-core matmul (one launch; K splits reduced in
// the cluster).  Returns the number of kernels launched, or -1 on a host-side
// failure.
static int launch_matmul(const MatmulDesc& d, cudaStream_t s, int* err) {
  CUtensorMap ta, tb;
  if (!make_operand_map(&ta, d.A, d.a_kmajor, d.a_kmajor ? d.M : d.K, d.a_kmajor ? d.K : d.M, d.lda)) return -1;
  if (!make_operand_map(&tb, d.B, d.b_kmajor, d.b_kmajor ? d.N : d.K, d.b_kmajor ? d.K : d.N, d.ldb)) return -1;
  int splits = choose_splits(d.M, d.N, d.K);
  tc::Params p;
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.a_kmajor = d.a_kmajor;
  p.b_kmajor = d.b_kmajor;
  p.k_tiles = ceil_div(d.K, tc::BK);
  p.kt_per_split = ceil_div(p.k_tiles, splits);
  p.epi = d.epi;
  p.splits = splits;
  p.err = err;
  const long long tiles = (long long)ceil_div(d.M, tc::BM) * ceil_div(d.N, tc::BN);
  const int num_sms = dev_info().num_sms;
  if (splits == 1 && tiles > num_sms) {
    // more tiles than SMs: one persistent CTA per SM walks them
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_sms);
    cfg.blockDim = dim3(tc::pers::THREADS);
    cfg.dynamicSmemBytes = tc::pers::SMEM_BYTES;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = g_pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, tc::gemm_tf32x3_persistent_kernel, ta, tb, p) != cudaSuccess) return -1;
    return 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ceil_div(d.N, tc::BN), ceil_div(d.M, tc::BM), splits);
  cfg.blockDim = dim3(tc::THREADS);
  cfg.dynamicSmemBytes = tc::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = splits;
  cfg.attrs = g_pdl ? attr : attr + 1;
  cfg.numAttrs = (g_pdl ? 1 : 0) + (splits > 1 ? 1 : 0);
  if (cudaLaunchKernelEx(&cfg, tc::gemm_tf32x3_kernel, ta, tb, p) != cudaSuccess) return -1;
  return 1;
}

// Tensor map of a bf16 operand stored as `outer` rows of pitch `ld` elements
// with `inner` valid contiguous elements per row, 128-byte swizzle.  K-major
// boxes are 64 (K) x box_rows; MN-major boxes are 64 (MN) x 64 (K).
// Out-of-range elements load as zero.
static int make_bf16_map(CUtensorMap* tm, const uint16_t* base, int kmajor, long long outer, long long inner,
                         long long ld, int box_rows) {
  if (!get_encoder()) return 0;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box_k[2] = {(cuuint32_t)tcb::BK, (cuuint32_t)box_rows};
  cuuint32_t box_mn[2] = {(cuuint32_t)tcb::MN_BOX, (cuuint32_t)tcb::BK};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, (void*)base, dims, strides,
                              kmajor ? box_k : box_mn, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}


// More epilogue warps for the GELU, GELU' and residual epilogues when the
// product has at most 20 K tiles (K <= 1280: the K = C products of the GPT-2
// shapes), where the epilogue, not the main loop, sets the pace.
constexpr int HEAVY_EPI_MAX_KTILES = 20;

template <int BN, int OP, int EG>
static void launch_bf16_cfg(const CUtensorMap& ta, const CUtensorMap& tb, const tcb::Params& p, int grid, cudaStream_t s) {
  using CF = tcb::Cfg<BN, OP, EG>;
  launch_k(tcb::gemm_bf16_kernel<BN, OP, EG>, grid, CF::THREADS, (size_t)CF::SMEM_BYTES, s, ta, tb, p);
}

template <int BN, int OP>
static void launch_bf16_op(const CUtensorMap& ta, const CUtensorMap& tb, const tcb::Params& p, int grid, cudaStream_t s) {
  if constexpr (tcb::heavy_epilogue(OP)) {
    if (p.k_tiles <= HEAVY_EPI_MAX_KTILES) {
      launch_bf16_cfg<BN, OP, tcb::heavy_epilogue_groups(OP)>(ta, tb, p, grid, s);
      return;
    }
  }
  launch_bf16_cfg<BN, OP, 2>(ta, tb, p, grid, s);
}

template <int BN>
static void launch_bf16_kernel(const CUtensorMap& ta, const CUtensorMap& tb, const tcb::Params& p, int grid,
                               cudaStream_t s) {
  switch (p.epi.epi) {
    case EPI_BIAS: launch_bf16_op<BN, EPI_BIAS>(ta, tb, p, grid, s); break;
    case EPI_BIAS_RESID: launch_bf16_op<BN, EPI_BIAS_RESID>(ta, tb, p, grid, s); break;
    case EPI_BIAS_GELU: launch_bf16_op<BN, EPI_BIAS_GELU>(ta, tb, p, grid, s); break;
    case EPI_DGELU: launch_bf16_op<BN, EPI_DGELU>(ta, tb, p, grid, s); break;
    case EPI_ACCUM: launch_bf16_op<BN, EPI_ACCUM>(ta, tb, p, grid, s); break;
    case EPI_LOGITS: launch_bf16_op<BN, EPI_LOGITS>(ta, tb, p, grid, s); break;
    default: launch_bf16_op<BN, EPI_STORE>(ta, tb, p, grid, s); break;
  }
}

// Raises the dynamic shared-memory limit of every epilogue instantiation.
template <int BN, int OP>
static cudaError_t set_bf16_smem_op() {
  const cudaFuncAttribute a = cudaFuncAttributeMaxDynamicSharedMemorySize;
  cudaError_t e = cudaFuncSetAttribute(tcb::gemm_bf16_kernel<BN, OP, 2>, a, tcb::Cfg<BN, OP, 2>::SMEM_BYTES);
  if constexpr (tcb::heavy_epilogue(OP)) {
    constexpr int EG = tcb::heavy_epilogue_groups(OP);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(tcb::gemm_bf16_kernel<BN, OP, EG>, a, tcb::Cfg<BN, OP, EG>::SMEM_BYTES);
  }
  return e;
}

template <int BN>
static cudaError_t set_bf16_smem() {
  cudaError_t e = set_bf16_smem_op<BN, EPI_STORE>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_BIAS>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_BIAS_RESID>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_BIAS_GELU>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_DGELU>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_ACCUM>();
  if (e == cudaSuccess) e = set_bf16_smem_op<BN, EPI_LOGITS>();
  return e;
}

// Output tiles and K splits of the persistent bf16 matmul.  A 128 x 256
// tile does its work at a higher rate than two 128 x 128 ones (which also
// read A twice); 128 x 128 tiles halve the K splits (and their partial-tile
// traffic) needed to fill the SMs.  K is split only when the tiles do not fill
// the SMs, keeping at least four 64-wide K tiles per split; never for the
// epilogues that take column sums or row statistics (no_split).
struct Bf16Plan {
  int BN, splits;
};

// Relative time of a plan: the waves of (tile, split) units times the K tiles
// each unit walks, a 128-wide tile's K tile costing 0.625 of a 256-wide one
// (half the MMA work at about 0.8 of the rate), a 192-wide one 0.88 of it, plus the last arrival's
// reduction of the fp32 partials (3 or 1.5 K-tile times per split).  The
// constants are fitted to the kernel timed alone on the GPT-2 product shapes.
static double bf16_plan_cost(int M, int N, int K, int BN, int splits, int num_sms) {
  const long long tiles = (long long)ceil_div(M, tcb::BM) * ceil_div(N, BN);
  const int kt = ceil_div(K, tcb::BK), per = ceil_div(kt, splits);
  const long long waves = (tiles * splits + num_sms - 1) / num_sms;
  const double c = BN == 256 ? 1.0 : (BN == 192 ? 0.88 : 0.625), r = BN * 3.0 / 256.0;
  return (double)waves * per * c + (splits > 1 ? splits * r : 0.0);
}

// The K split of a BN-wide plan: s = min(SMs / tiles, K tiles / 4) for grids
// below one wave with at least 8 K tiles, lowered until the fp32 partials fit
// the workspace, then rounded to equal K ranges.
static int bf16_splits(int M, int N, int K, int BN, bool no_split, long long ws_floats, int num_sms) {
  const long long tiles = (long long)ceil_div(M, tcb::BM) * ceil_div(N, BN);
  const int kt = ceil_div(K, tcb::BK);
  if (no_split || tiles >= num_sms || kt < 8) return 1;
  int s = (int)(num_sms / tiles);
  s = s < kt / 4 ? s : kt / 4;
  while (s > 1 && (long long)s * M * N > ws_floats) s--;
  if (s < 1) s = 1;
  return ceil_div(kt, ceil_div(kt, s));
}

// 256-wide tiles when they fill at least two thirds of a wave, else 128-wide,
// with the K split above.  Another width (128, 192 or 256, the 192-wide one
// unless excluded) or a smaller split replaces that plan only when its
// modelled time is at least 10% lower.  On the GPT-2 shapes this turns the
// 124M weight gradients into 256-wide tiles split in two (one wave of
// 256-wide tiles instead of one of 128-wide tiles), and the 774M products
// with N = 1280 at B*T = 4096 into 192-wide tiles (224 tiles in two waves
// instead of 160 256-wide ones, the second nearly empty).
static Bf16Plan plan_bf16(int M, int N, int K, bool no_split, long long ws_floats, int num_sms, bool allow192 = true) {
  const long long tiles256 = (long long)ceil_div(M, tcb::BM) * ceil_div(N, 256);
  const int BN = (N > 128 && 3 * tiles256 >= 2 * num_sms) ? 256 : 128;
  const Bf16Plan plan = {BN, bf16_splits(M, N, K, BN, no_split, ws_floats, num_sms)};
  const double base = bf16_plan_cost(M, N, K, plan.BN, plan.splits, num_sms);
  const int kt = ceil_div(K, tcb::BK);
  double best = base;
  Bf16Plan alt = plan;
  for (int bn = 128; bn <= 256; bn += 64) {
    if (bn > 128 && N <= 128) break;
    if (bn == 192 && !allow192) continue;
    const int smax = bf16_splits(M, N, K, bn, no_split, ws_floats, num_sms);
    for (int s = 1; s <= smax; s++) {
      const int sp = ceil_div(kt, ceil_div(kt, s));
      const double c = bf16_plan_cost(M, N, K, bn, sp, num_sms);
      if (c < best) {
        best = c;
        alt = {bn, sp};
      }
    }
  }
  return best <= 0.9 * base ? alt : plan;
}

// Launches the persistent bf16 tensor-core matmul.  Returns 1, or -1 on a
// host-side failure.
static int launch_matmul_bf16(const MatmulDesc& d, float* ws, int* tile_ctr, int* err, cudaStream_t s,
                              long long ws_floats = SPLITK_WS_FLOATS) {
  if (!d.Abf || !d.Bbf) return -1;
  // column sums and the row statistics are taken in the warp epilogue, which a K split bypasses
  const bool no_split = d.epi.colsum || d.epi.epi == EPI_LOGITS;
  // the LM head's row statistics are per half of a 256-wide tile
  const Bf16Plan plan = plan_bf16(d.M, d.N, d.K, no_split, ws_floats, dev_info().num_sms, d.epi.epi != EPI_LOGITS);
  const int BN = plan.BN;
  CUtensorMap ta, tb;
  if (!make_bf16_map(&ta, d.Abf, d.a_kmajor, d.a_kmajor ? d.M : d.K, d.a_kmajor ? d.K : d.M, d.lda, tcb::BM))
    return -1;
  if (!make_bf16_map(&tb, d.Bbf, d.b_kmajor, d.b_kmajor ? d.N : d.K, d.b_kmajor ? d.K : d.N, d.ldb, BN)) return -1;
  tcb::Params p;
  p.M = d.M;
  p.N = d.N;
  p.K = d.K;
  p.a_kmajor = d.a_kmajor;
  p.b_kmajor = d.b_kmajor;
  p.splits = plan.splits;
  if (d.epi.epi == EPI_LOGITS && (!d.epi.vec4 || !d.epi.Cbf || d.epi.C)) return -1;
  if (d.epi.colsum && (!d.epi.vec4 || d.N % 32 || (d.epi.ldcs & 3) || ((uintptr_t)d.epi.colsum & 15))) return -1;
  p.k_tiles = ceil_div(d.K, tcb::BK);
  p.kt_per_split = ceil_div(p.k_tiles, p.splits);
  p.tiles_m = ceil_div(d.M, tcb::BM);
  p.tiles_n = ceil_div(d.N, BN);
  p.units = p.tiles_m * p.tiles_n * p.splits;
  p.epi = d.epi;
  p.epi.fast = 1;  // bf16 outputs: GELU through the hardware tanh approximation
  p.partial = p.splits > 1 ? ws : nullptr;
  p.tile_ctr = tile_ctr;
  p.err = err;
  const int nsm = dev_info().num_sms;
  int grid = p.units < nsm ? p.units : nsm;
  if (BN == 256) launch_bf16_kernel<256>(ta, tb, p, grid, s);
  else if (BN == 192) launch_bf16_kernel<192>(ta, tb, p, grid, s);
  else launch_bf16_kernel<128>(ta, tb, p, grid, s);
  return 1;
}

static int matmul(gpt2_t* m, const MatmulDesc& d, cudaStream_t st = nullptr) {
  if (d.epi.colsum && m->cfg.gemm_precision != GPT2_PREC_BF16) {  // fused column sums: bf16 kernel only
    m->poisoned = GPT2_ERR_CUDA;
    return GPT2_ERR_CUDA;
  }
  if (!st) st = m->stream;
  timer_begin(m, TK_GEMM, 2.0 * d.M * (double)d.N * d.K);
  // the weight-gradient side stream has a split-K workspace of its own
  const bool on_w = st == m->side_w && m->splitk_w;
  int n = m->cfg.gemm_precision == GPT2_PREC_BF16
              ? launch_matmul_bf16(d, on_w ? m->splitk_w : m->splitk, on_w ? m->tilectr_w : m->tilectr, m->err, st)
                                                  : launch_matmul(d, st, m->err);
  timer_end(m, TK_GEMM);
  if (n < 0) {
    m->poisoned = GPT2_ERR_CUDA;
    return GPT2_ERR_CUDA;
  }
  m->launches += n;
  return GPT2_OK;
}

static EpiArgs epi_args(float* C, long long ldc, int epi, const float* bias = nullptr, const float* R = nullptr,
                        long long ldr = 0, float* pre = nullptr, long long ldpre = 0, uint16_t* Cbf = nullptr,
                        long long ldcbf = 0) {
  EpiArgs e;
  e.C = C; e.ldc = ldc; e.bias = bias; e.R = R; e.ldr = ldr; e.pre = pre; e.ldpre = ldpre; e.epi = epi;
  e.Cbf = Cbf; e.ldcbf = ldcbf; e.fast = 0;
  e.colsum = nullptr; e.ldcs = 0;
  e.targets = nullptr; e.V = 0; e.xstats = nullptr; e.ldxs = 0; e.tlogit = nullptr;
  e.pre_bf = nullptr; e.Rbf = nullptr;
  uintptr_t addr = (uintptr_t)C | (uintptr_t)bias | (uintptr_t)R | (uintptr_t)pre | (uintptr_t)Cbf;
  e.vec4 = (addr & 15) == 0 && (ldc & 3) == 0 && (ldr & 3) == 0 && (ldpre & 3) == 0 && (ldcbf & 7) == 0;
  return e;
}

// A matmul operand: the fp32 array and, for bf16 matmuls, its bf16 copy.
struct Opnd {
  const float* f;
  const uint16_t* h;
};

// linear layer y = x W^T + b with x (N, IC), W (OC, IC); ybf: optional bf16 copy of y
static void mm_forward(gpt2_t* m, float* out, uint16_t* outbf, Opnd x, Opnd W, const float* bias, int N, int IC,
                       int OC, int epi, const float* R, float* pre, uint16_t* pre_bf = nullptr) {
  MatmulDesc d = {N, OC, IC, x.f, IC, 1, W.f, IC, 1, epi_args(out, OC, epi, bias, R, OC, pre, OC, outbf, OC), x.h, W.h};
  d.epi.pre_bf = pre_bf;
  if ((uintptr_t)pre_bf & 7) d.epi.vec4 = 0;
  matmul(m, d);
}

// dx = dy W (times gelu'(pre) when pre != NULL); colsum: optional 32-row
// column partial sums of dx (bf16 matmuls), leading dimension IC
// ---- the backward's side stream -------------------------------------------
// side_fork: the side stream continues after everything enqueued so far on
// the main stream; returns the event side_done records at the end of the side
// work.  side_wait: the main stream waits for a pending side reader of a
// buffer before overwriting it.  side_join: the main stream waits for all side
// work.  The kernel timer brackets launches on the main stream only, so under
// it (and on a handle without a side stream) everything stays on the main
// stream.
static bool side_on(const gpt2_t* m) { return m->side && m->timer_kind == TK_NONE; }

static int side_fork(gpt2_t* m, cudaStream_t* st) {
  *st = m->stream;  // also the stream of the failure path below
  if (!side_on(m)) return -1;
  const int f = m->sev_next, d = (m->sev_next + 1) % SIDE_EVENTS;
  m->sev_next = (m->sev_next + 2) % SIDE_EVENTS;
  cudaError_t e = cudaEventRecord(m->sev[f], m->stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(m->side, m->sev[f], 0);
  if (e != cudaSuccess) {
    fprintf(stderr, "gpt2b300: %s (side stream fork)\n", cudaGetErrorString(e));
    m->poisoned = GPT2_ERR_CUDA;
    return -1;
  }
  *st = m->side;
  return d;
}

static int side_done(gpt2_t* m, int d, int* reader) {
  if (d < 0) return GPT2_OK;
  CCHECK(m, cudaEventRecord(m->sev[d], m->side));
  m->side_last = d;
  if (reader) *reader = d;
  return GPT2_OK;
}

static int side_wait(gpt2_t* m, int* reader) {
  if (*reader >= 0) CCHECK(m, cudaStreamWaitEvent(m->stream, m->sev[*reader], 0));
  *reader = -1;
  return GPT2_OK;
}

static int side_join(gpt2_t* m) {
  if (m->side_last >= 0) CCHECK(m, cudaStreamWaitEvent(m->stream, m->sev[m->side_last], 0));
  if (m->side_w_last >= 0) CCHECK(m, cudaStreamWaitEvent(m->stream, m->sev[m->side_w_last], 0));
  m->side_last = m->rd_scratch = m->rd_dfch = m->rd_dqkv = -1;
  m->side_w_last = m->wd_dres = m->wd_dfch = m->wd_dqkv = -1;
  return GPT2_OK;
}

static void mm_dx(gpt2_t* m, float* dx, uint16_t* dxbf, Opnd dy, Opnd W, int N, int IC, int OC, const float* pre,
                  float* colsum = nullptr, const uint16_t* pre_bf = nullptr) {
  MatmulDesc d = {N,    IC,   OC,   dy.f, OC, 1, W.f, IC, 0,
                  epi_args(dx, IC, (pre || pre_bf) ? EPI_DGELU : EPI_STORE, nullptr, pre, IC, nullptr, 0, dxbf, IC),
                  dy.h, W.h};
  d.epi.Rbf = pre_bf;
  if (pre_bf) d.epi.ldr = IC;
  if ((uintptr_t)pre_bf & 7) d.epi.vec4 = 0;
  d.epi.colsum = colsum;
  d.epi.ldcs = IC;
  if (colsum == m->scratch) side_wait(m, &m->rd_scratch);
  matmul(m, d);
}

// dW += dy^T x  (dW = dy^T x in the fused step, whose gradients start from zero)
static void mm_dw(gpt2_t* m, float* dW, Opnd dy, Opnd x, int N, int IC, int OC) {
  MatmulDesc d = {OC, IC, N, dy.f, OC, 0, x.f, IC, 0, epi_args(dW, IC, m->grad_accumulate ? EPI_ACCUM : EPI_STORE),
                  dy.h, x.h};
  matmul(m, d);
}

// The same on the weight-gradient side stream: it starts after
// everything enqueued so far on the main stream, and *reader records when it
// has finished reading dy (x is a per-layer activation nothing overwrites
// during the backward).
static void mm_dw_side(gpt2_t* m, float* dW, Opnd dy, Opnd x, int N, int IC, int OC, int* reader) {
  // fp32 reduces K splits inside a cluster; bf16 needs the side stream's own workspace
  if (!side_on(m) || !m->side_w || (m->cfg.gemm_precision != GPT2_PREC_FP32 && !m->splitk_w)) {
    mm_dw(m, dW, dy, x, N, IC, OC);
    return;
  }
  const int f = m->sev_next, d = (m->sev_next + 1) % SIDE_EVENTS;
  m->sev_next = (m->sev_next + 2) % SIDE_EVENTS;
  if (cudaEventRecord(m->sev[f], m->stream) != cudaSuccess || cudaStreamWaitEvent(m->side_w, m->sev[f], 0) != cudaSuccess) {
    m->poisoned = GPT2_ERR_CUDA;
    return;
  }
  MatmulDesc md = {OC, IC, N, dy.f, OC, 0, x.f, IC, 0, epi_args(dW, IC, m->grad_accumulate ? EPI_ACCUM : EPI_STORE),
                   dy.h, x.h};
  matmul(m, md, m->side_w);
  if (cudaEventRecord(m->sev[d], m->side_w) != cudaSuccess) {
    m->poisoned = GPT2_ERR_CUDA;
    return;
  }
  m->side_w_last = d;
  *reader = d;
}

// db += column sums of dy (N, OC): chunks of BIAS_MIN_ROWS rows summed by
// one thread per column, then the chunk partials finished in a fixed order.
// Up to BIAS_DIRECT_ROWS rows the finishing kernel sums dy's rows itself
// (32 warps, each striding over the rows): one launch instead of two.
#define BIAS_DIRECT_ROWS 2048
// The direct form runs on the side stream; *reader records when it has
// finished reading dy.
static void bias_grad(gpt2_t* m, float* db, const float* dy, int N, int OC, int* reader) {
  if (N <= BIAS_DIRECT_ROWS) {
    cudaStream_t st;
    const int d = side_fork(m, &st);
    launch_k(col_finish_kernel, ceil_div(OC, 32), COLF_WARPS * 32, 0, st, db, db, db, OC, dy, N, OC,
             m->grad_accumulate);
    side_done(m, d, reader);
    m->launches++;
    return;
  }
  side_wait(m, &m->rd_scratch);
  const int rows = BIAS_MIN_ROWS, chunks = ceil_div(N, rows);
  launch_k(col_partial_kernel, dim3(ceil_div(OC, 256), chunks), 256, 0, m->stream, dy, N, OC, OC, rows, m->scratch);
  launch_k(col_finish_kernel, ceil_div(OC, 32), COLF_WARPS * 32, 0, m->stream, db, db, db, OC, m->scratch, chunks,
           OC, m->grad_accumulate);
  m->launches += 2;
}

// db (+)= the sums of the nrows column-partial rows (OC columns) a matmul or
// attention epilogue left in m->scratch
static_assert(BIAS_MIN_ROWS == 32, "the scratch is sized in 32-row column-sum blocks");
static void bias_finish(gpt2_t* m, float* db, int nrows, int OC) {
  cudaStream_t st;
  const int d = side_fork(m, &st);
  launch_k(col_finish_kernel, ceil_div(OC, 32), COLF_WARPS * 32, 0, st, db, db, db, OC, m->scratch, nrows, OC,
           m->grad_accumulate);
  side_done(m, d, &m->rd_scratch);
  m->launches++;
}

template <typename K>
static K ln_pick(int C, K k1, K k2, K k4, K k6, K k8, K k10) {
  const int v = ceil_div(C, 128);
  return v <= 1 ? k1 : v <= 2 ? k2 : v <= 4 ? k4 : v <= 6 ? k6 : v <= 8 ? k8 : k10;
}

// Layernorm forward blocks: four warps (rows).  Block residency is counted in
// whole blocks, so small blocks keep more rows in flight: at C = 1280 (72
// registers a thread) seven 4-warp blocks fit an SM, 1036 on the GPU, and a
// 4096-row launch runs in one wave, where 8-warp blocks (three an SM) left
// 68 blocks for a second one.
#define LNF_WARPS 4

static void ln_forward(gpt2_t* m, float* y, uint16_t* ybf, float* mean, float* rstd, const float* x, const float* w,
                       const float* b, int N) {
  int C = m->cfg.channels;
  // read x; write y (fp32) and/or its bf16 copy; mean and rstd
  timer_begin(m, TK_LAYERNORM, (4.0 * C + (y ? 4.0 * C : 0.0) + (ybf ? 2.0 * C : 0.0) + 8.0) * N);
  if (m->cfg.llama) {  // RMSNorm: no mean, no shift
    auto k = ln_pick(C, layernorm_fwd_kernel<1, true>, layernorm_fwd_kernel<2, true>, layernorm_fwd_kernel<4, true>,
                     layernorm_fwd_kernel<6, true>, layernorm_fwd_kernel<8, true>, layernorm_fwd_kernel<10, true>);
    launch_k(k, ceil_div(N, LNF_WARPS), LNF_WARPS * 32, 0, m->stream, y, ybf, mean, rstd, x, w, (const float*)nullptr, N,
             C);
  } else {
    auto k = ln_pick(C, layernorm_fwd_kernel<1, false>, layernorm_fwd_kernel<2, false>, layernorm_fwd_kernel<4, false>,
                     layernorm_fwd_kernel<6, false>, layernorm_fwd_kernel<8, false>, layernorm_fwd_kernel<10, false>);
    launch_k(k, ceil_div(N, LNF_WARPS), LNF_WARPS * 32, 0, m->stream, y, ybf, mean, rstd, x, w, b, N, C);
  }
  timer_end(m, TK_LAYERNORM);
  m->launches++;
}

// layernorm backward: dx += ...; dw, db (+)= the parameter gradients; when
// dxsum != NULL also dxsum (+)= the column sums of the updated dx -- the bias
// gradient of the linear layer whose output gradient dx is.
static void ln_backward(gpt2_t* m, float* dx, uint16_t* dxbf, float* dw, float* db, float* dxsum, const float* dy,
                        const float* x, const float* w, const float* mean, const float* rstd, int N) {
  int C = m->cfg.channels;
  const int nb = ceil_div(N, LNB_WARPS);  // one row per warp
  const bool rms = m->cfg.llama != 0;        // RMSNorm: dw only (no shift, no linear biases)
  const int nout = rms ? 1 : (dxsum ? 3 : 2);
  // read dy, x, mean, rstd and dx; write dx (and its bf16 copy)
  timer_begin(m, TK_LAYERNORM, (16.0 * C + 8.0 + (dxbf ? 2.0 * C : 0.0)) * N);
  side_wait(m, &m->rd_scratch);  // the partials below overwrite the scratch
  if (dx == m->dres) side_wait(m, &m->wd_dres);
  const int wds = dxsum ? 1 : 0;
  int nparts = nb;  // partial rows the column finish sums
  const int nsm = dev_info().num_sms;
  if (nb > 2 * nsm) {
    // many rows: one block per SM walking the rows, one partial row per block
    const int W = ln_pick(C, LnbStride<1>::WARPS, LnbStride<2>::WARPS, LnbStride<4>::WARPS, LnbStride<6>::WARPS,
                          LnbStride<8>::WARPS, LnbStride<10>::WARPS);
    const size_t smem = (size_t)W * nout * C * sizeof(float);
    nparts = nsm;
    if (rms) {
      auto k = ln_pick(C, layernorm_bwd_stride_kernel<1, true>, layernorm_bwd_stride_kernel<2, true>,
                       layernorm_bwd_stride_kernel<4, true>, layernorm_bwd_stride_kernel<6, true>,
                       layernorm_bwd_stride_kernel<8, true>, layernorm_bwd_stride_kernel<10, true>);
      launch_k(k, nsm, W * 32, smem, m->stream, dx, dxbf, m->scratch, dy, x, w, mean, rstd, N, C, 0);
    } else {
      auto k = ln_pick(C, layernorm_bwd_stride_kernel<1, false>, layernorm_bwd_stride_kernel<2, false>,
                       layernorm_bwd_stride_kernel<4, false>, layernorm_bwd_stride_kernel<6, false>,
                       layernorm_bwd_stride_kernel<8, false>, layernorm_bwd_stride_kernel<10, false>);
      launch_k(k, nsm, W * 32, smem, m->stream, dx, dxbf, m->scratch, dy, x, w, mean, rstd, N, C, wds);
    }
  } else {
    const size_t smem = (size_t)LNB_WARPS * nout * C * sizeof(float);
    if (rms) {
      auto k = ln_pick(C, layernorm_bwd_kernel<1, true>, layernorm_bwd_kernel<2, true>, layernorm_bwd_kernel<4, true>,
                       layernorm_bwd_kernel<6, true>, layernorm_bwd_kernel<8, true>, layernorm_bwd_kernel<10, true>);
      launch_k(k, nb, LNB_WARPS * 32, smem, m->stream, dx, dxbf, m->scratch, dy, x, w, mean, rstd, N, C, 0);
    } else {
      auto k = ln_pick(C, layernorm_bwd_kernel<1, false>, layernorm_bwd_kernel<2, false>, layernorm_bwd_kernel<4, false>,
                       layernorm_bwd_kernel<6, false>, layernorm_bwd_kernel<8, false>, layernorm_bwd_kernel<10, false>);
      launch_k(k, nb, LNB_WARPS * 32, smem, m->stream, dx, dxbf, m->scratch, dy, x, w, mean, rstd, N, C, wds);
    }
  }
  // dw[c] (+)= sum_b partial[b][c], db[c] (+)= sum_b partial[b][C + c], dxsum[c] (+)= ...[2C + c]
  cudaStream_t st;
  const int d = side_fork(m, &st);
  launch_k(col_finish_kernel, ceil_div(nout * C, 32), COLF_WARPS * 32, 0, st, dw, db, dxsum, C, m->scratch, nparts,
           nout * C, m->grad_accumulate);
  side_done(m, d, &m->rd_scratch);
  timer_end(m, TK_LAYERNORM);
  m->launches += 2;
}

// Tensor map of an fp32 matrix stored as `outer` rows of pitch `ld` elements
// with `inner` valid columns: 32 x 64 boxes (128-byte rows) with the 128-byte
// swizzle, the tile format of the short-sequence fp32 attention.
static int make_f32_box64_map(CUtensorMap* tm, const float* base, long long outer, long long inner, long long ld) {
  if (!get_encoder()) return 0;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld * sizeof(float)};
  cuuint32_t box[2] = {32, 64};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, (void*)base, dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 operands, head size 64, T <= 64: the 3xTF32 tensor-core kernels
static bool attn_tf32_path(int bf, int hs, int T) { return !bf && hs == atf::HS && T <= atf::T_MAX; }

// Causal attention forward: the tensor-core kernel for bf16 operands with
// head size 64 and T % 128 == 0, else the CUDA-core kernel (the template
// argument is the number of head dimensions each lane holds, hs <= 32 * ND).
// Returns the number of launches, or -1 on a host-side failure.
static int launch_attn_fwd(float* atty, uint16_t* attybf, float* lse, const float* qkv, const uint16_t* qkv_bf, int B,
                           int T, int C, int NH, int bf, int* err, cudaStream_t s) {
  const int hs = C / NH;
  if (bf && qkv_bf && hs == tca::HS && T % tca::BQ == 0) {
    // qkv with 128-row boxes (Q tiles) and 64-row boxes (K, V tiles)
    CUtensorMap tq, tkv;
    if (!make_bf16_map(&tq, qkv_bf, 1, (long long)B * T, 3LL * C, 3LL * C, tca::BQ)) return -1;
    if (!make_bf16_map(&tkv, qkv_bf, 1, (long long)B * T, 3LL * C, 3LL * C, tca::fwd::FKV)) return -1;
    tca::Params p;
    p.B = B; p.T = T; p.C = C; p.NH = NH;
    p.scale = 1.0f / sqrtf((float)hs);
    p.y = atty; p.ybf = attybf; p.lse = lse; p.err = err;
    // persistent: two CTAs on each SM walk the (query tile, head, batch) items
    const long long items = (long long)(T / tca::BQ) * NH * B, slots = 2LL * dev_info().num_sms;
    launch_k(tca::attn_fwd_tc_kernel, (int)(items < slots ? items : slots), tca::THREADS, tca::fwd::SMEM_BYTES, s, tq,
             tkv, p);
    return 1;
  }
  if (attn_tf32_path(bf, hs, T)) {  // fp32, short sequences: one CTA per (head, batch), 3xTF32 products
    CUtensorMap tm;
    if (!make_f32_box64_map(&tm, qkv, (long long)B * T, 3LL * C, 3LL * C)) return -1;
    atf::Params p = {};
    p.B = B; p.T = T; p.C = C; p.NH = NH;
    p.scale = 1.0f / sqrtf((float)hs);
    p.qkv = qkv; p.out = atty; p.out_bf = attybf; p.lse = lse; p.err = err;
    launch_k(atf::attn_fwd_tf32_kernel, dim3(NH, B), atf::THREADS, atf::FWD_SMEM, s, tm, p);
    return 1;
  }
  if (T <= atts::T_MAX && hs == atts::HS) {  // short sequences: one CTA per (batch, head)
    launch_k(atts::attn_fwd_small_kernel, dim3(NH, B), atts::THREADS, atts::FWD_SMEM, s, atty, attybf, lse, qkv, B, T,
             C, NH, bf);
    return 1;
  }
  const dim3 g(ceil_div(T, ATT_ROWS), NH, B);
  const size_t sm = att_smem_fwd(hs);
  if (hs <= 32) launch_k(attn_fwd_simt_kernel<1>, g, ATT_ROWS * 32, sm, s, atty, attybf, lse, qkv, B, T, C, NH, bf);
  else if (hs <= 64) launch_k(attn_fwd_simt_kernel<2>, g, ATT_ROWS * 32, sm, s, atty, attybf, lse, qkv, B, T, C, NH, bf);
  else launch_k(attn_fwd_simt_kernel<4>, g, ATT_ROWS * 32, sm, s, atty, attybf, lse, qkv, B, T, C, NH, bf);
  return 1;
}

static void attn_forward(gpt2_t* m, float* atty, uint16_t* attybf, float* lse, const float* qkv,
                         const uint16_t* qkv_bf, int B, int T, int bf) {
  int C = m->cfg.channels, NH = m->cfg.num_heads, hs = C / NH;
  timer_begin(m, TK_ATTN_FWD, 4.0 * (double)B * NH * T * (T + 1) / 2.0 * hs);
  int n = launch_attn_fwd(atty, attybf, lse, qkv, qkv_bf, B, T, C, NH, bf, m->err, m->stream);
  timer_end(m, TK_ATTN_FWD);
  if (n < 0) {
    m->poisoned = GPT2_ERR_CUDA;
    return;
  }
  m->launches += n;
}

// Causal attention backward into dqkv (and its bf16 copy): D = rowsum(dy o y),
// then the tensor-core dK/dV and dQ kernels (bf16, hs = 64, T % 128 == 0) or
// the CUDA-core kernels.  Returns the number of launches, or -1.
static int launch_attn_bwd(float* dqkv, uint16_t* dqkv_bf, float* D, const float* dy, const uint16_t* dy_bf,
                           const float* qkv, const uint16_t* qkv_bf, const float* atty, const float* lse, int B, int T,
                           int C, int NH, int bf, int* err, cudaStream_t s, float* colsum = nullptr,
                           const uint16_t* atty_bf = nullptr) {
  const int hs = C / NH;
  const int grid = ceil_div((long long)B * NH * T * 32, 256);
  const bool tc_path = bf && qkv_bf && dy_bf && hs == tca::HS && T % tca::BQ == 0;
  if (!tc_path && attn_tf32_path(bf, hs, T)) {  // fp32, short sequences: dQ and dK/dV kernels, 3xTF32 products
    if (!dqkv || colsum) return -1;
    CUtensorMap tq, td, ty;
    if (!make_f32_box64_map(&tq, qkv, (long long)B * T, 3LL * C, 3LL * C)) return -1;
    if (!make_f32_box64_map(&td, dy, (long long)B * T, C, C)) return -1;
    if (!make_f32_box64_map(&ty, atty, (long long)B * T, C, C)) return -1;
    atf::Params p = {};
    p.B = B; p.T = T; p.C = C; p.NH = NH;
    p.scale = 1.0f / sqrtf((float)hs);
    p.qkv = qkv; p.dy = dy; p.y = atty; p.out = dqkv; p.out_bf = dqkv_bf; p.lse = (float*)lse; p.err = err;
    launch_k(atf::attn_bwd_tf32_kernel, dim3(NH, B, 2), atf::THREADS, atf::BWD_SMEM, s, tq, td, ty, p);
    return 1;
  }
  if (!tc_path && T <= atts::T_MAX && hs == atts::HS) {  // short sequences: one launch, D formed in the kernel
    if (!dqkv || colsum) return -1;
    launch_k(atts::attn_bwd_small_kernel, dim3(NH, B), atts::THREADS, atts::BWD_SMEM, s, dqkv, dqkv_bf, qkv, dy, atty,
             lse, B, T, C, NH, bf);
    return 1;
  }
  // D holds 2 B NH T floats: the (-lse log2 e, -D) pairs of the tensor-core path
  const int ldg = ceil_div((long long)B * T, tca::LD_WARPS);
  if (tc_path && atty_bf && C <= 1024)  // from the bf16 copies of dO and y (the fp32 ones are not written)
    launch_k(tca::attn_bwd_ld_bf16_kernel<8>, ldg, tca::LD_WARPS * 32, 0, s, (float2*)D, lse, dy_bf, atty_bf, B, T, C);
  else if (tc_path && atty_bf && C <= 2048)
    launch_k(tca::attn_bwd_ld_bf16_kernel<16>, ldg, tca::LD_WARPS * 32, 0, s, (float2*)D, lse, dy_bf, atty_bf, B, T, C);
  else if (tc_path && C <= 1024)
    launch_k(tca::attn_bwd_ld_kernel<8>, ldg, tca::LD_WARPS * 32, 0, s, (float2*)D, lse, dy, atty, B, T, C);
  else if (tc_path && C <= 2048)
    launch_k(tca::attn_bwd_ld_kernel<16>, ldg, tca::LD_WARPS * 32, 0, s, (float2*)D, lse, dy, atty, B, T, C);
  else
    launch_k(attn_bwd_D_kernel, grid, 256, 0, s, tc_path ? nullptr : D, tc_path ? (float2*)D : nullptr, lse, dy, atty,
             B, T, C, NH);
  if (tc_path) {
    // qkv and dO with 128-row boxes (whole tiles) and 64-row boxes (sub-tiles)
    CUtensorMap tq, tq64, td, td64;
    if (!make_bf16_map(&tq, qkv_bf, 1, (long long)B * T, 3LL * C, 3LL * C, tca::BQ)) return -1;
    if (!make_bf16_map(&tq64, qkv_bf, 1, (long long)B * T, 3LL * C, 3LL * C, tca::SUB)) return -1;
    if (!make_bf16_map(&td, dy_bf, 1, (long long)B * T, C, C, tca::BQ)) return -1;
    if (!make_bf16_map(&td64, dy_bf, 1, (long long)B * T, C, C, tca::SUB)) return -1;
    tca::BwdParams p;
    p.B = B; p.T = T; p.C = C; p.NH = NH;
    p.scale = 1.0f / sqrtf((float)hs);
    p.LD = (const float2*)D; p.dqkv = dqkv; p.dqkv_bf = dqkv_bf; p.colsum = colsum; p.err = err;
    // persistent: one CTA per SM walks the (tile, head, batch) items
    const long long items = (long long)(T / tca::BQ) * NH * B, nsm = dev_info().num_sms;
    const int g = (int)(items < nsm ? items : nsm);
    launch_k(tca::attn_bwd_dkv_tc_kernel, g, tca::DKV_THREADS, tca::dkv::SMEM_BYTES, s, tq, tq64, td64, p);
    launch_k(tca::attn_bwd_dq_tc_kernel, g, tca::DQ_THREADS, tca::dqk::SMEM_BYTES, s, tq, tq64, td, p);
    return 3;
  }
  if (!dqkv || colsum) return -1;  // the CUDA-core kernels store fp32 dqkv only
  const dim3 g(ceil_div(T, ATT_ROWS), NH, B);
  const size_t sq = att_smem_fwd(hs), skv = att_smem_dkv(hs);
  if (hs <= 32) {
    launch_k(attn_bwd_dq_kernel<1>, g, ATT_ROWS * 32, sq, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
    launch_k(attn_bwd_dkv_kernel<1>, g, ATT_ROWS * 32, skv, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
  } else if (hs <= 64) {
    launch_k(attn_bwd_dq_kernel<2>, g, ATT_ROWS * 32, sq, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
    launch_k(attn_bwd_dkv_kernel<2>, g, ATT_ROWS * 32, skv, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
  } else {
    launch_k(attn_bwd_dq_kernel<4>, g, ATT_ROWS * 32, sq, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
    launch_k(attn_bwd_dkv_kernel<4>, g, ATT_ROWS * 32, skv, s, dqkv, dqkv_bf, qkv, dy, lse, D, B, T, C, NH, bf);
  }
  return 3;
}

// fuse_bias: the tensor-core kernels leave the 128-row column sums of dqkv in
// m->scratch (the QKV bias gradient's first stage) and skip the fp32 dqkv,
// which nothing else reads in bf16 precision
static void attn_backward(gpt2_t* m, const float* qkv, const uint16_t* qkv_bf, const float* atty,
                          const uint16_t* atty_bf, const float* lse, int B, int T, int bf, bool fuse_bias) {
  int C = m->cfg.channels, NH = m->cfg.num_heads, hs = C / NH;
  side_wait(m, &m->rd_dqkv);
  side_wait(m, &m->wd_dqkv);
  if (fuse_bias) side_wait(m, &m->rd_scratch);
  timer_begin(m, TK_ATTN_BWD, 8.0 * (double)B * NH * T * (T + 1) / 2.0 * hs);
  int n = launch_attn_bwd(fuse_bias ? nullptr : m->dqkv, m->dqkv_bf, m->attD, m->datty, m->datty_bf, qkv, qkv_bf, atty,
                          lse, B, T, C, NH, bf, m->err, m->stream, fuse_bias ? m->scratch : nullptr, atty_bf);
  timer_end(m, TK_ATTN_BWD);
  if (n < 0) {
    m->poisoned = GPT2_ERR_CUDA;
    return;
  }
  m->launches += n;
}

// Dynamic shared memory limits of the large-smem kernels.  They apply per
// device, so they are set once for each device the library is used on, with
// that device current.
static int set_kernel_attributes() {
  const int dev = current_device();
  if (dev < 0) return GPT2_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo* di = &g_dev[dev];
  if (di->attr) return di->attr > 0 ? GPT2_OK : GPT2_ERR_CUDA;
  {
    cudaError_t e = cudaFuncSetAttribute(sort_tokens_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SORT_MAX * (int)sizeof(uint32_t));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc::gemm_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, tc::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tc::gemm_tf32x3_persistent_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tc::pers::SMEM_BYTES);
    if (e == cudaSuccess) e = query_cluster_limits(dev, di);
    if (e == cudaSuccess) e = set_bf16_smem<256>();
    if (e == cudaSuccess) e = set_bf16_smem<192>();
    if (e == cudaSuccess) e = set_bf16_smem<128>();
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tca::attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tca::fwd::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tca::attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tca::dkv::SMEM_BYTES);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(tca::attn_bwd_dq_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               tca::dqk::SMEM_BYTES);
    // layernorm backward: 8 rows x 3C floats of shared memory (C <= 1280)
    const int lnb = LNB_WARPS * 3 * 32 * 4 * LN_MAXV4_LIMIT * (int)sizeof(float);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<2, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<2, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<6, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<6, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<8, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<8, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<10, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(layernorm_bwd_kernel<10, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, lnb);
    // the row-walking variant: LnbStride::WARPS slots of 3 x 128 V4 floats
#define LNB_STRIDE_ATTR(V4)                                                                                   \
  if (e == cudaSuccess)                                                                                       \
    e = cudaFuncSetAttribute(layernorm_bwd_stride_kernel<V4, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                             LnbStride<V4>::WARPS * 3 * 128 * V4 * (int)sizeof(float));                       \
  if (e == cudaSuccess)                                                                                       \
    e = cudaFuncSetAttribute(layernorm_bwd_stride_kernel<V4, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,  \
                             LnbStride<V4>::WARPS * 3 * 128 * V4 * (int)sizeof(float));
    LNB_STRIDE_ATTR(1) LNB_STRIDE_ATTR(2) LNB_STRIDE_ATTR(4) LNB_STRIDE_ATTR(6) LNB_STRIDE_ATTR(8) LNB_STRIDE_ATTR(10)
#undef LNB_STRIDE_ATTR
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(atf::attn_fwd_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)atf::FWD_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(atf::attn_bwd_tf32_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)atf::BWD_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(atts::attn_fwd_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)atts::FWD_SMEM);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(atts::attn_bwd_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)atts::BWD_SMEM);
    // CUDA-core attention: up to head size 128
    const int f = (int)att_smem_fwd(128), kv = (int)att_smem_dkv(128);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_fwd_simt_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_fwd_simt_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_fwd_simt_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dq_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dq_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dq_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dkv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dkv_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(attn_bwd_dkv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, kv);
    if (e != cudaSuccess) {
      fprintf(stderr, "gpt2b300: cudaFuncSetAttribute failed on device %d: %s\n", dev, cudaGetErrorString(e));
      cudaGetLastError();
      di->attr = -1;
    } else {
      di->attr = 1;
    }
  }
  return di->attr > 0 ? GPT2_OK : GPT2_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// the three phases
// ---------------------------------------------------------------------------
// Per-layer views of the activation arena (rows strided by maxB * maxT).  The
// bf16 copies exist only for bf16 matmuls (NULL otherwise).
struct LayerActs {
  const float* x;  // layer input (residual stream)
  float *ln1, *qkv, *atty, *lse, *res2, *ln2, *fch, *fchg, *res3;
  float *ln1_mean, *ln1_rstd, *ln2_mean, *ln2_rstd;
  uint16_t *ln1_bf, *qkv_bf, *atty_bf, *ln2_bf, *fchg_bf;
  uint16_t* fch_bf;  // the pre-activation in bf16 (bf16 matmuls; fch is then NULL)
};

static LayerActs layer_acts(gpt2_t* m, int l) {
  const size_t cap = (size_t)m->maxB * m->maxT, C = m->cfg.channels, NH = m->cfg.num_heads;
  LayerActs a;
  a.x = l == 0 ? m->encoded : m->res3 + (size_t)(l - 1) * cap * C;
  a.ln1 = m->ln1 + l * cap * C;
  a.qkv = m->qkv + l * cap * 3 * C;
  a.atty = m->atty + l * cap * C;
  a.lse = m->lse + l * cap * NH;
  a.res2 = m->res2 + l * cap * C;
  a.ln2 = m->ln2 + l * cap * C;
  a.fch = m->fch + l * cap * 4 * C;
  a.fchg = m->fchg + l * cap * 4 * C;
  a.res3 = m->res3 + l * cap * C;
  a.ln1_mean = m->ln1_mean + l * cap;
  a.ln1_rstd = m->ln1_rstd + l * cap;
  a.ln2_mean = m->ln2_mean + l * cap;
  a.ln2_rstd = m->ln2_rstd + l * cap;
  const bool bf = m->params_bf != nullptr;
  a.ln1_bf = bf ? m->ln1_bf + l * cap * C : nullptr;
  a.qkv_bf = bf ? m->qkv_bf + l * cap * 3 * C : nullptr;
  a.atty_bf = bf ? m->atty_bf + l * cap * C : nullptr;
  a.ln2_bf = bf ? m->ln2_bf + l * cap * C : nullptr;
  a.fchg_bf = bf ? m->fchg_bf + l * cap * 4 * C : nullptr;
  a.fch_bf = bf ? (uint16_t*)m->fch + l * cap * 4 * C : nullptr;
  if (bf) a.fch = nullptr;
  return a;
}

// fp32 parameter tensor i (+ offset) and its bf16 copy
static Opnd wparam(gpt2_t* m, int i, size_t off) {
  Opnd o;
  o.f = m->P[i] + off;
  o.h = m->params_bf ? m->params_bf + (m->P[i] - m->params) + off : nullptr;
  return o;
}

static int enqueue_forward(gpt2_t* m, const int* d_in, const int* d_tgt, int B, int T, int validate) {
  const gpt2_config& c = m->cfg;
  int L = c.num_layers, C = c.channels, V = c.vocab_size, Vp = c.padded_vocab_size;
  int N = B * T;
  cudaStream_t s = m->stream;
  int bf = c.gemm_precision == GPT2_PREC_BF16;
  const size_t CC = (size_t)C * C;
  if (validate) {
    launch_k(validate_tokens_kernel, grid_for(N, 256, 64), 256, 0, s, d_in, d_tgt, N, V, m->err);
    m->launches++;
  }
  // reads a wte row and a wpe row, writes one row per token
  timer_begin(m, TK_ENCODER, (c.llama ? 8.0 : 12.0) * C * N);
  launch_k(encoder_fwd_kernel, grid_for((long long)N * C / 4, 256), 256, 0, s, m->encoded, d_in, m->P[P_WTE],
           c.llama ? (const float*)nullptr : m->P[P_WPE], N, T, C, V);
  timer_end(m, TK_ENCODER);
  m->launches++;
  // bf16 matmuls read only the bf16 copies: the fp32 layernorm outputs, the
  // fp32 GELU output and (with the tensor-core attention) the fp32 qkv are
  // then not written at all
  const bool tc_attn = bf && C / c.num_heads == tca::HS && T % tca::BQ == 0;
  // the Llama-style variant has no linear biases: its matmuls add a zero vector
  auto bias = [&](int which, size_t off) -> const float* { return c.llama ? m->zero_bias : m->P[which] + off; };
  for (int l = 0; l < L; l++) {
    LayerActs a = layer_acts(m, l);
    ln_forward(m, bf ? nullptr : a.ln1, a.ln1_bf, a.ln1_mean, a.ln1_rstd, a.x, m->P[P_LN1W] + (size_t)l * C,
               m->P[P_LN1B] + (size_t)l * C, N);
    // the rotary embedding reads and rewrites the fp32 q and k, so the variant keeps fp32 qkv
    mm_forward(m, tc_attn && !c.llama ? nullptr : a.qkv, a.qkv_bf, {a.ln1, a.ln1_bf}, wparam(m, P_QKVW, l * 3 * CC),
               bias(P_QKVB, (size_t)l * 3 * C), N, C, 3 * C, EPI_BIAS, nullptr, nullptr);
    if (c.llama) {
      launch_k(rope_kernel, grid_for((long long)N * C / 2, 256), 256, 0, s, a.qkv, a.qkv_bf, (const float2*)m->rope, B,
               T, C, c.num_heads, 0);
      m->launches++;
    }
    // with the tensor-core attention only the bf16 copy of its output is read
    attn_forward(m, tc_attn ? nullptr : a.atty, a.atty_bf, a.lse, a.qkv, a.qkv_bf, B, T, bf);
    mm_forward(m, a.res2, nullptr, {a.atty, a.atty_bf}, wparam(m, P_ATTPROJW, l * CC), bias(P_ATTPROJB, (size_t)l * C),
               N, C, C, EPI_BIAS_RESID, a.x, nullptr);
    ln_forward(m, bf ? nullptr : a.ln2, a.ln2_bf, a.ln2_mean, a.ln2_rstd, a.res2, m->P[P_LN2W] + (size_t)l * C,
               m->P[P_LN2B] + (size_t)l * C, N);
    mm_forward(m, bf ? nullptr : a.fchg, a.fchg_bf, {a.ln2, a.ln2_bf}, wparam(m, P_FCW, l * 4 * CC),
               bias(P_FCB, (size_t)l * 4 * C), N, C, 4 * C, EPI_BIAS_GELU, nullptr, a.fch, a.fch_bf);
    mm_forward(m, a.res3, nullptr, {a.fchg, a.fchg_bf}, wparam(m, P_FCPROJW, l * 4 * CC),
               bias(P_FCPROJB, (size_t)l * C), N, 4 * C, C, EPI_BIAS_RESID, a.res2, nullptr);
  }
  LayerActs last = layer_acts(m, L - 1);
  ln_forward(m, bf ? nullptr : m->lnf, m->lnf_bf, m->lnf_mean, m->lnf_rstd, last.res3, m->P[P_LNFW], m->P[P_LNFB], N);
  // bf16 matmuls with targets: the LM head stores its logits in bf16 and
  // leaves the rows' softmax statistics and the targets' fp32 logits, so the
  // cross-entropy reads the logits once (bf16) instead of twice (fp32)
  const bool xbf = bf && d_tgt;
  if (xbf) {
    const Opnd wte = wparam(m, P_WTE, 0);
    MatmulDesc d = {N, Vp, C, m->lnf, C, 1, wte.f, C, 1,
                    epi_args(nullptr, Vp, EPI_LOGITS, nullptr, nullptr, 0, nullptr, 0, m->logits_bf, Vp), m->lnf_bf,
                    wte.h};
    d.epi.targets = d_tgt;
    d.epi.V = V;
    d.epi.xstats = m->xstats;
    d.epi.ldxs = (int)xstats_pitch(Vp);
    d.epi.tlogit = m->tlogit;
    matmul(m, d);
  } else {
    mm_forward(m, m->logits, nullptr, {m->lnf, m->lnf_bf}, wparam(m, P_WTE, 0), nullptr, N, C, Vp, EPI_STORE, nullptr,
               nullptr);
  }
  m->logits_in_bf = xbf ? 1 : 0;
  if (xbf) {
    // the LM head's tile width, as its launch chose it (EPI_LOGITS: no split)
    const int bn = plan_bf16(N, Vp, C, true, SPLITK_WS_FLOATS, dev_info().num_sms, false).BN;
    const int nblk = ceil_div(Vp, bn / 2), ldxs = (int)xstats_pitch(Vp);
    // reads the bf16 logits and the statistics, writes the bf16 dlogits
    timer_begin(m, TK_XENT, (double)N * (4.0 * Vp + 8.0 * nblk + 8.0));
    launch_k(xent_bf16_kernel, N, XENT_BF_THREADS, 0, s, m->dlogits_bf, m->losses, (const uint16_t*)m->logits_bf,
             (const float2*)m->xstats, nblk, ldxs, (const float*)m->tlogit, d_tgt, V, Vp, 1.0f / (float)N);
    timer_end(m, TK_XENT);
    launch_k(mean_kernel, 1, 1024, 0, s, m->losses, N, m->loss);
    m->launches += 2;
  } else if (d_tgt) {
    timer_begin(m, TK_XENT, 8.0 * (double)N * Vp);
    launch_k(xent_fused_kernel, N, XENT_THREADS, 0, s, m->dlogits, (uint16_t*)nullptr, m->losses, m->logits, d_tgt, V,
             Vp, 1.0f / (float)N);
    timer_end(m, TK_XENT);
    launch_k(mean_kernel, 1, 1024, 0, s, m->losses, N, m->loss);
    m->launches += 2;
  }
  KCHECK(m);
  m->B = B;
  m->T = T;
  m->have_targets = d_tgt != nullptr;
  m->fwd_done = 1;
  return GPT2_OK;
}

static int update_layer(gpt2_t* m, int l);
static int mark_touched_rows(gpt2_t* m, int N);
static int update_wte_untouched(gpt2_t* m);

static int enqueue_backward(gpt2_t* m) {
  const gpt2_config& c = m->cfg;
  int L = c.num_layers, C = c.channels, Vp = c.padded_vocab_size;
  int B = m->B, T = m->T, N = B * T;
  cudaStream_t s = m->stream;
  int bf = c.gemm_precision == GPT2_PREC_BF16;
  const size_t CC = (size_t)C * C;
  float** P = m->P;
  float** G = m->G;
  const Opnd dres = {m->dres, m->dres_bf}, dfch = {m->dfch, m->dfch_bf}, dqkv = {m->dqkv, m->dqkv_bf};
  // the Llama-style variant has no biases (and no bias gradients) and no position table
  const bool ll = c.llama != 0;
  // the fused column sums need 32-column-aligned rows of 16-byte-aligned floats
  const bool fuse_fcb = bf && !ll && (4 * C) % 32 == 0;
  // the tensor-core attention backward (bf16, hs = 64, T % 128 == 0) takes the QKV bias column sums
  const bool tc_attn = bf && C / c.num_heads == tca::HS && T % tca::BQ == 0;  // the tensor-core attention
  const bool fuse_qkvb = tc_attn && !ll;
  auto gbias = [&](int which, size_t off) -> float* { return ll ? nullptr : G[which] + off; };
  if (m->upd_layers) {
    int rc = mark_touched_rows(m, N);
    if (rc) return rc;
  }
  // LM head (tied to wte): dlnf = dlogits wte; dwte += dlogits^T lnf
  mm_dx(m, m->dln, nullptr, {m->dlogits, m->dlogits_bf}, wparam(m, P_WTE, 0), N, C, Vp, nullptr);
  mm_dw(m, G[P_WTE], {m->dlogits, m->dlogits_bf}, {m->lnf, m->lnf_bf}, N, C, Vp);
  if (m->upd_layers) {  // nothing later reads wte, and the untouched rows' gradients are final
    int rc = update_wte_untouched(m);
    if (rc) return rc;
  }
  CCHECK(m, cudaMemsetAsync(m->dres, 0, (size_t)N * C * sizeof(float), s));
  LayerActs last = layer_acts(m, L - 1);
  // the column sums of this dres are the last layer's MLP output-projection bias gradient
  ln_backward(m, m->dres, m->dres_bf, G[P_LNFW], G[P_LNFB], gbias(P_FCPROJB, (size_t)(L - 1) * C), m->dln, last.res3,
              P[P_LNFW], m->lnf_mean, m->lnf_rstd, N);
  for (int l = L - 1; l >= 0; l--) {
    LayerActs a = layer_acts(m, l);
    // MLP output projection: res3 = res2 + fchg fcprojw^T + fcprojb
    mm_dw_side(m, G[P_FCPROJW] + l * 4 * CC, dres, {a.fchg, a.fchg_bf}, N, 4 * C, C, &m->wd_dres);
    // (its bias gradient came with the layernorm backward that produced dres)
    // x gelu'(fch).  bf16: only the bf16 copy of dfch is stored; the MLP input
    // bias gradient comes from column sums taken in the same epilogue
    side_wait(m, &m->rd_dfch);  // dfch is overwritten here
    side_wait(m, &m->wd_dfch);
    mm_dx(m, bf && (fuse_fcb || ll) ? nullptr : m->dfch, m->dfch_bf, dres, wparam(m, P_FCPROJW, l * 4 * CC), N, 4 * C, C,
          a.fch, fuse_fcb ? m->scratch : nullptr, a.fch_bf);
    // MLP input projection: fch = ln2 fcw^T + fcb
    mm_dw_side(m, G[P_FCW] + l * 4 * CC, dfch, {a.ln2, a.ln2_bf}, N, C, 4 * C, &m->wd_dfch);
    if (fuse_fcb) bias_finish(m, G[P_FCB] + (size_t)l * 4 * C, ceil_div(N, 32), 4 * C);
    else if (!ll) bias_grad(m, G[P_FCB] + (size_t)l * 4 * C, m->dfch, N, 4 * C, &m->rd_dfch);
    mm_dx(m, m->dln, nullptr, dfch, wparam(m, P_FCW, l * 4 * CC), N, C, 4 * C, nullptr);
    ln_backward(m, m->dres, m->dres_bf, G[P_LN2W] + (size_t)l * C, G[P_LN2B] + (size_t)l * C,
                gbias(P_ATTPROJB, (size_t)l * C), m->dln, a.res2, P[P_LN2W] + (size_t)l * C, a.ln2_mean, a.ln2_rstd, N);
    // attention output projection: res2 = x + atty attprojw^T + attprojb
    mm_dw_side(m, G[P_ATTPROJW] + l * CC, dres, {a.atty, a.atty_bf}, N, C, C, &m->wd_dres);
    // (the tensor-core attention backward reads only the bf16 copy of datty)
    mm_dx(m, tc_attn ? nullptr : m->datty, m->datty_bf, dres, wparam(m, P_ATTPROJW, l * CC), N, C, C, nullptr);
    // attention
    attn_backward(m, a.qkv, a.qkv_bf, tc_attn ? nullptr : a.atty, a.atty_bf, a.lse, B, T, bf, fuse_qkvb);
    if (ll) {  // q and k were rotated after the matmul: turn their gradients back (the transpose)
      launch_k(rope_kernel, grid_for((long long)N * C / 2, 256), 256, 0, s, m->dqkv, m->dqkv_bf, (const float2*)m->rope,
               B, T, C, c.num_heads, 1);
      m->launches++;
    }
    // qkv projection: qkv = ln1 qkvw^T + qkvb
    mm_dw_side(m, G[P_QKVW] + l * 3 * CC, dqkv, {a.ln1, a.ln1_bf}, N, C, 3 * C, &m->wd_dqkv);
    if (fuse_qkvb) bias_finish(m, G[P_QKVB] + (size_t)l * 3 * C, N / tca::BQ, 3 * C);
    else if (!ll) bias_grad(m, G[P_QKVB] + (size_t)l * 3 * C, m->dqkv, N, 3 * C, &m->rd_dqkv);
    mm_dx(m, m->dln, nullptr, dqkv, wparam(m, P_QKVW, l * 3 * CC), N, C, 3 * C, nullptr);
    // below layer 0 this dres is the previous layer's MLP output gradient
    ln_backward(m, m->dres, m->dres_bf, G[P_LN1W] + (size_t)l * C, G[P_LN1B] + (size_t)l * C,
                l > 0 ? gbias(P_FCPROJB, (size_t)(l - 1) * C) : nullptr, m->dln, a.x, P[P_LN1W] + (size_t)l * C,
                a.ln1_mean, a.ln1_rstd, N);
    // every gradient of layer l is complete once the work enqueued so far is
    if (m->upd_layers) {
      int rc = update_layer(m, l);
      if (rc) return rc;
    }
  }
  // embeddings: positions sorted by (id, position), then one CTA per id's run
  const int V = c.vocab_size;
  if (N <= SORT_BITONIC_MAX) {
    size_t smem = 1;
    while ((int)smem < N) smem <<= 1;
    launch_k(sort_tokens_kernel, 1, 1024, smem * sizeof(uint32_t), s, (const int*)m->tokens, N, V, m->sorted);
    m->launches++;
  } else {  // stable radix sort by the id's low byte, then its high byte
    const int nch = ceil_div(N, RADIX_CHUNK);
    for (int pass = 0; pass < 2; pass++) {
      const uint32_t* src = pass ? m->sort_tmp : nullptr;
      uint32_t* dst = pass ? m->sorted : m->sort_tmp;
      launch_k(radix_hist_kernel, nch, RADIX_THREADS, 0, s, (const int*)m->tokens, V, src, N, 8 * pass, m->radix_hist);
      launch_k(radix_scan_kernel, 1, 1024, 0, s, m->radix_hist, 256 * nch);
      launch_k(radix_scatter_kernel, nch, RADIX_THREADS, 0, s, (const int*)m->tokens, V, src, N, 8 * pass,
               (const int*)m->radix_hist, dst);
      m->launches += 3;
    }
  }
  launch_k(run_starts_kernel, 1, 1024, 0, s, (const uint32_t*)m->sorted, (const int*)m->tokens, V, N, m->runs,
           m->nruns);
  launch_k(wte_grad_kernel, dim3(grid_for(N, 1, 4 * 148), ceil_div(C, 128)), WTE_WARPS * 32, 0, s, G[P_WTE], m->dres,
           (const uint32_t*)m->sorted, (const int*)m->tokens, V, (const int*)m->runs, (const int*)m->nruns, N, C);
  m->launches += 2;
  if (!ll) {
    launch_k(wpe_grad_kernel, grid_for((long long)T * C / 4, 256), 256, 0, s, G[P_WPE], m->dres, B, T, C,
             m->grad_accumulate);
    m->launches++;
  }
  KCHECK(m);
  return side_join(m);  // every gradient is complete on the main stream from here on
}

// AdamW hyper-parameters live in device memory so that a captured step can
// be replayed with a new step number: {lr, b1, b2, eps, wd, 1/(1-b1^t), 1/(1-b2^t)}.
static int write_hparams(gpt2_t* m, float lr, float b1, float b2, float eps, float wd, int t) {
  double c1 = 1.0 - pow((double)b1, t), c2 = 1.0 - pow((double)b2, t);
  float h[8] = {lr, b1, b2, eps, wd, (float)(1.0 / c1), (float)(1.0 / c2), 0.f};
  // pageable source: the copy is staged before the call returns, so h may go out of scope
  CCHECK(m, cudaMemcpyAsync(m->hparams, h, sizeof(h), cudaMemcpyHostToDevice, m->stream));
  return GPT2_OK;
}

// AdamW over k pieces (element offset into the flat buffers, element count) in
// one launch, on stream st.
static int launch_adamw(gpt2_t* m, const long long* off, const long long* cnt, int k, cudaStream_t st) {
  AdamSegs sg = {};
  long long tot = 0;
  for (int i = 0; i < k; i++) {
    if (cnt[i] <= 0) continue;  // the Llama-style variant's empty tensors
    if (sg.n == ADAMW_MAX_SEGS || (off[i] & 3) || (cnt[i] & 3)) {
      m->poisoned = GPT2_ERR_CUDA;
      return GPT2_ERR_CUDA;
    }
    sg.off4[sg.n] = off[i] / 4;
    tot += cnt[i] / 4;
    sg.end4[sg.n++] = tot;
  }
  if (!sg.n) return GPT2_OK;
  const bool on_main = st == m->stream;
  if (on_main) timer_begin(m, TK_ADAMW, 4.0 * tot * (28.0 + (m->params_bf ? 2.0 : 0.0)));
  launch_k(adamw_kernel, grid_for(tot, 256, 148 * 8), 256, 0, st, m->params, (const float*)m->grads, m->m, m->v, sg,
           (const float*)m->hparams, m->params_bf);
  if (on_main) timer_end(m, TK_ADAMW);
  m->launches++;
  KCHECK(m);
  return GPT2_OK;
}

static long long poff(const gpt2_t* m, int i) { return (long long)(m->P[i] - m->params); }

// AdamW of every parameter (gpt2_update)
static int enqueue_update(gpt2_t* m) {
  const long long off = 0, cnt = m->np;
  return launch_adamw(m, &off, &cnt, 1, m->stream);
}

// The update side stream continues after everything enqueued so far on the
// main stream and both gradient side streams; returns the stream to launch
// on (the main stream when side streams are off).
static cudaStream_t upd_fork(gpt2_t* m) {
  if (!side_on(m) || !m->side_u) return m->stream;
  const int f = m->sev_next;
  m->sev_next = (m->sev_next + 1) % SIDE_EVENTS;
  if (cudaEventRecord(m->sev[f], m->stream) != cudaSuccess || cudaStreamWaitEvent(m->side_u, m->sev[f], 0) != cudaSuccess ||
      (m->side_last >= 0 && cudaStreamWaitEvent(m->side_u, m->sev[m->side_last], 0) != cudaSuccess) ||
      (m->side_w_last >= 0 && cudaStreamWaitEvent(m->side_u, m->sev[m->side_w_last], 0) != cudaSuccess)) {
    m->poisoned = GPT2_ERR_CUDA;
    return m->stream;
  }
  return m->side_u;
}

static int upd_done(gpt2_t* m, cudaStream_t st) {
  if (st == m->stream) return m->poisoned ? m->poisoned : GPT2_OK;
  const int d = m->sev_next;
  m->sev_next = (m->sev_next + 1) % SIDE_EVENTS;
  CCHECK(m, cudaEventRecord(m->sev[d], st));
  m->side_u_last = d;
  return GPT2_OK;
}

// AdamW of layer l's twelve tensors, once their gradients are complete.
// Called by the fused step's backward after layer l's last kernel.
static int update_layer(gpt2_t* m, int l) {
  static const int T[12] = {P_LN1W, P_LN1B, P_QKVW, P_QKVB, P_ATTPROJW, P_ATTPROJB,
                            P_LN2W, P_LN2B, P_FCW,  P_FCB,  P_FCPROJW,  P_FCPROJB};
  const long long L = m->cfg.num_layers;
  long long off[12], cnt[12];
  for (int i = 0; i < 12; i++) {
    cnt[i] = m->psize[T[i]] / L;
    off[i] = poff(m, T[i]) + l * cnt[i];
  }
  cudaStream_t st = upd_fork(m);
  int rc = launch_adamw(m, off, cnt, 12, st);
  return rc ? rc : upd_done(m, st);
}

// The fused step's wte rows: those no token of the batch touches have their
// final gradient once the LM head's weight gradient is done, so they are
// updated right after it (part 1); the rows the tokens touch also get the
// embedding gradient, at the end of the backward (part 2, update_rest).
static int mark_touched_rows(gpt2_t* m, int N) {
  CCHECK(m, cudaMemsetAsync(m->rowmask, 0, (size_t)m->cfg.padded_vocab_size, m->stream));
  launch_k(mark_rows_kernel, grid_for(N, 256, 64), 256, 0, m->stream, (const int*)m->tokens, N, m->cfg.vocab_size,
           m->rowmask);
  m->launches++;
  KCHECK(m);
  return GPT2_OK;
}

static int update_wte_untouched(gpt2_t* m) {
  cudaStream_t st = upd_fork(m);
  const int C = m->cfg.channels, Vp = m->cfg.padded_vocab_size;
  const bool on_main = st == m->stream;
  if (on_main) timer_begin(m, TK_ADAMW, 4.0 * (double)Vp * C * (7.0 + (m->params_bf ? 0.5 : 0.0)));
  launch_k(adamw_rows_kernel, grid_for((long long)Vp * C / 4, 256, 148 * 8), 256, 0, st, m->params,
           (const float*)m->grads, m->m, m->v, poff(m, P_WTE), Vp, C, (const uint8_t*)m->rowmask, 0,
           (const float*)m->hparams, m->params_bf);
  if (on_main) timer_end(m, TK_ADAMW);
  m->launches++;
  KCHECK(m);
  return upd_done(m, st);
}

// The rest of the fused step's AdamW, after joining the earlier updates: the
// wte rows the batch's tokens touch (one CTA per sorted token key; the CTA at
// the first key of each id updates its row), then wpe and the final
// layernorm.
static int update_rest(gpt2_t* m, int N) {
  if (m->side_u_last >= 0) CCHECK(m, cudaStreamWaitEvent(m->stream, m->sev[m->side_u_last], 0));
  m->side_u_last = -1;
  const int C = m->cfg.channels;
  timer_begin(m, TK_ADAMW, 0.0);  // the touched rows' bytes are not known on the host: counted as 0
  launch_k(adamw_sorted_rows_kernel, grid_for(N, 1, 4 * 148), 256, 0, m->stream, m->params, (const float*)m->grads,
           m->m, m->v, poff(m, P_WTE), C, (const uint32_t*)m->sorted, (const int*)m->tokens, m->cfg.vocab_size,
           (const int*)m->runs, (const int*)m->nruns, (const float*)m->hparams, m->params_bf);
  timer_end(m, TK_ADAMW);
  m->launches++;
  KCHECK(m);
  const long long off[3] = {poff(m, P_WPE), poff(m, P_LNFW), poff(m, P_LNFB)};
  const long long cnt[3] = {m->psize[P_WPE], m->psize[P_LNFW], m->psize[P_LNFB]};
  return launch_adamw(m, off, cnt, 3, m->stream);
}

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
EXPORT size_t gpt2_arena_bytes(const gpt2_config* cfg, int maxB, int maxT) {
  if (!config_ok(cfg) || !shape_ok(cfg, maxB, maxT)) return 0;
  Plan p;
  return plan_arena(cfg, maxB, maxT, &p);
}

EXPORT const char* gpt2_status_string(int s) {
  switch (s) {
    case GPT2_OK: return "ok";
    case GPT2_ERR_ARG: return "invalid argument";
    case GPT2_ERR_SHAPE: return "invalid shape (B, T outside the handle's limits)";
    case GPT2_ERR_TOKEN_RANGE: return "token id outside [0, vocab_size)";
    case GPT2_ERR_STATE: return "backward without a forward that had targets";
    case GPT2_ERR_ARENA: return "arena too small or misaligned";
    case GPT2_ERR_CUDA: return "CUDA error (handle poisoned)";
    case GPT2_ERR_DEVICE_TIMEOUT: return "device-side wait timed out (handle poisoned)";
    case GPT2_WARN_NONFINITE: return "loss is not finite";
    default: return "unknown status";
  }
}

static void carve(gpt2_t* m) {
  char* a = m->arena;
  const Plan& p = m->plan;
  m->params = (float*)(a + p.params);
  m->grads = (float*)(a + p.grads);
  m->m = (float*)(a + p.m);
  m->v = (float*)(a + p.v);
  m->params_bf = m->cfg.gemm_precision == GPT2_PREC_BF16 ? (uint16_t*)(a + p.params_bf) : nullptr;
  long long off = 0;
  for (int i = 0; i < NUM_PARAMS; i++) {
    m->P[i] = m->params + off;
    m->G[i] = m->grads + off;
    off += m->psize[i];
  }
#define CARVE(f) m->f = (decltype(m->f))(a + p.f)
  CARVE(encoded); CARVE(ln1); CARVE(ln1_mean); CARVE(ln1_rstd); CARVE(qkv); CARVE(atty); CARVE(lse);
  CARVE(res2); CARVE(ln2); CARVE(ln2_mean); CARVE(ln2_rstd); CARVE(fch); CARVE(fchg); CARVE(res3);
  CARVE(lnf); CARVE(lnf_mean); CARVE(lnf_rstd); CARVE(logits); CARVE(dlogits); CARVE(losses); CARVE(loss);
  CARVE(dres); CARVE(dln); CARVE(datty); CARVE(dqkv); CARVE(dfch); CARVE(attD); CARVE(scratch); CARVE(sorted);
  CARVE(sort_tmp); CARVE(radix_hist); CARVE(runs);
  m->nruns = m->runs + (size_t)m->maxB * m->maxT;
  CARVE(tokens); CARVE(targets); CARVE(err); CARVE(hparams); CARVE(splitk); CARVE(tilectr);
  CARVE(splitk_w); CARVE(tilectr_w);
  if (m->cfg.gemm_precision != GPT2_PREC_BF16) m->splitk_w = nullptr, m->tilectr_w = nullptr;
#undef CARVE
#define CARVE_BF(f) m->f = m->params_bf ? (uint16_t*)(a + p.f) : nullptr
  CARVE_BF(ln1_bf); CARVE_BF(qkv_bf); CARVE_BF(atty_bf); CARVE_BF(ln2_bf); CARVE_BF(fchg_bf); CARVE_BF(lnf_bf); CARVE_BF(dlogits_bf);
  CARVE_BF(dres_bf); CARVE_BF(dfch_bf); CARVE_BF(dqkv_bf); CARVE_BF(datty_bf); CARVE_BF(logits_bf);
  m->xstats = m->params_bf ? (float2*)(a + p.xstats) : nullptr;
  m->tlogit = m->params_bf ? (float*)(a + p.tlogit) : nullptr;
  m->rowmask = (uint8_t*)(a + p.rowmask);
  m->rope = m->cfg.llama ? (float2*)(a + p.rope) : nullptr;
  m->zero_bias = m->cfg.llama ? (float*)(a + p.zero_bias) : nullptr;
#undef CARVE_BF
}

static int init_params(gpt2_t* m, uint64_t seed) {
  const gpt2_config& c = m->cfg;
  double proj = 0.02 / sqrt(2.0 * c.num_layers);
  long long off = 0;
  for (int i = 0; i < NUM_PARAMS; i++) {
    long long n = m->psize[i], nrand = 0;
    double stdv = 0.0;
    float fill = 0.f;
    switch (i) {
      case P_WTE: nrand = (long long)c.vocab_size * c.channels; stdv = 0.02; break;
      case P_WPE: case P_QKVW: case P_FCW: nrand = n; stdv = 0.02; break;
      case P_ATTPROJW: case P_FCPROJW: nrand = n; stdv = proj; break;
      case P_LN1W: case P_LN2W: case P_LNFW: fill = 1.f; break;
      default: break;
    }
    launch_k(init_tensor_kernel, grid_for(n, 256), 256, 0, m->stream, m->P[i], off, n, nrand, stdv, fill, seed);
    off += n;
  }
  KCHECK(m);
  return GPT2_OK;
}

static int refresh_bf16(gpt2_t* m) {
  if (!m->params_bf) return GPT2_OK;
  launch_k(to_bf16_kernel, grid_for(m->np, 256), 256, 0, m->stream, m->params, m->params_bf, m->np);
  KCHECK(m);
  return GPT2_OK;
}

EXPORT int gpt2_build(gpt2_t** out, const gpt2_config* cfg, uint64_t seed, int maxB, int maxT, void* dev_arena,
                      size_t arena_bytes, void* cuda_stream) {
  if (!out || !config_ok(cfg)) return GPT2_ERR_ARG;
  *out = nullptr;
  if (!shape_ok(cfg, maxB, maxT)) return GPT2_ERR_SHAPE;
  gpt2_t* m = (gpt2_t*)calloc(1, sizeof(gpt2_t));
  if (!m) return GPT2_ERR_ARG;
  m->grad_accumulate = 1;
  m->cfg = *cfg;
  m->maxB = maxB;
  m->maxT = maxT;
  m->np = param_count(cfg, m->psize);
  size_t need = plan_arena(cfg, maxB, maxT, &m->plan);
  m->stream = (cudaStream_t)cuda_stream;
  if (dev_arena) {
    if (arena_bytes < need || ((uintptr_t)dev_arena & 255)) {
      free(m);
      return GPT2_ERR_ARENA;
    }
    m->arena = (char*)dev_arena;
  } else {
    if (cudaMalloc((void**)&m->arena, need) != cudaSuccess) {
      cudaGetLastError();
      free(m);
      return GPT2_ERR_CUDA;
    }
    m->own_arena = 1;
  }
  carve(m);
  int rc;
  cudaError_t e;
  m->side_last = m->rd_scratch = m->rd_dfch = m->rd_dqkv = -1;
  m->side_w_last = m->wd_dres = m->wd_dfch = m->wd_dqkv = -1;
  m->side_u_last = -1;
  if (set_kernel_attributes() != GPT2_OK) {
    rc = GPT2_ERR_CUDA;
    goto fail;
  }
  if ((e = cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking)) != cudaSuccess) {
    m->side = nullptr;
    goto cuda_fail;
  }
  {
    int lo = 0, hi = 0;  // the weight-gradient side stream at the lowest priority
    if ((e = cudaDeviceGetStreamPriorityRange(&lo, &hi)) != cudaSuccess) goto cuda_fail;
    if ((e = cudaStreamCreateWithPriority(&m->side_w, cudaStreamNonBlocking, lo)) != cudaSuccess) {
      m->side_w = nullptr;
      goto cuda_fail;
    }
    if ((e = cudaStreamCreateWithPriority(&m->side_u, cudaStreamNonBlocking, lo)) != cudaSuccess) {
      m->side_u = nullptr;
      goto cuda_fail;
    }
  }
  for (int i = 0; i < SIDE_EVENTS; i++)
    if ((e = cudaEventCreateWithFlags(&m->sev[i], cudaEventDisableTiming)) != cudaSuccess) goto cuda_fail;
  if ((e = cudaMemsetAsync(m->grads, 0, m->np * sizeof(float), m->stream)) != cudaSuccess) goto cuda_fail;
  if ((e = cudaMemsetAsync(m->m, 0, m->np * sizeof(float), m->stream)) != cudaSuccess) goto cuda_fail;
  if ((e = cudaMemsetAsync(m->v, 0, m->np * sizeof(float), m->stream)) != cudaSuccess) goto cuda_fail;
  if ((e = cudaMemsetAsync(m->err, 0, sizeof(int), m->stream)) != cudaSuccess) goto cuda_fail;
  if ((e = cudaMemsetAsync(m->tilectr, 0, TILE_CTRS * sizeof(int), m->stream)) != cudaSuccess) goto cuda_fail;
  if (m->tilectr_w && (e = cudaMemsetAsync(m->tilectr_w, 0, TILE_CTRS * sizeof(int), m->stream)) != cudaSuccess)
    goto cuda_fail;
  if ((rc = init_params(m, seed)) != GPT2_OK) goto fail;
  if ((rc = refresh_bf16(m)) != GPT2_OK) goto fail;
  if (m->cfg.llama) {
    // rotary angles t * 10000^(-2i/hs) in double, stored as (cos, sin) floats:
    // accurate to float rounding even where t * frequency is ~1000 radians
    const int half = cfg->channels / cfg->num_heads / 2;
    std::vector<float2> tab((size_t)maxT * half);
    for (int t = 0; t < maxT; t++)
      for (int i = 0; i < half; i++) {
        const double theta = t * pow(10000.0, -2.0 * i / (2.0 * half));
        tab[(size_t)t * half + i] = make_float2((float)cos(theta), (float)sin(theta));
      }
    if ((e = cudaMemcpyAsync(m->rope, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice, m->stream)) !=
        cudaSuccess)
      goto cuda_fail;
    if ((e = cudaMemsetAsync(m->zero_bias, 0, 4 * (size_t)cfg->channels * sizeof(float), m->stream)) != cudaSuccess)
      goto cuda_fail;
    if ((e = cudaStreamSynchronize(m->stream)) != cudaSuccess) goto cuda_fail;  // tab is released on return
  }
  if ((e = cudaStreamSynchronize(m->stream)) != cudaSuccess) goto cuda_fail;
  *out = m;
  return GPT2_OK;
cuda_fail:
  fprintf(stderr, "gpt2b300: build failed: %s\n", cudaGetErrorString(e));
  cudaGetLastError();
  rc = GPT2_ERR_CUDA;
fail:
  for (int i = 0; i < SIDE_EVENTS; i++)
    if (m->sev[i]) cudaEventDestroy(m->sev[i]);
  if (m->side) cudaStreamDestroy(m->side);
  if (m->side_w) cudaStreamDestroy(m->side_w);
  if (m->side_u) cudaStreamDestroy(m->side_u);
  if (m->own_arena) cudaFree(m->arena);
  free(m);
  return rc;
}

EXPORT int gpt2_free(gpt2_t* m) {
  if (!m) return GPT2_ERR_ARG;
  cudaStreamSynchronize(m->stream);
  if (m->side) {
    cudaStreamSynchronize(m->side);
    cudaStreamDestroy(m->side);
  }
  if (m->side_w) {
    cudaStreamSynchronize(m->side_w);
    cudaStreamDestroy(m->side_w);
  }
  if (m->side_u) {
    cudaStreamSynchronize(m->side_u);
    cudaStreamDestroy(m->side_u);
  }
  for (int i = 0; i < SIDE_EVENTS; i++)
    if (m->sev[i]) cudaEventDestroy(m->sev[i]);
  if (m->gexec) cudaGraphExecDestroy(m->gexec);
  if (m->tev) {
    for (int i = 0; i < 2 * m->tcap; i++) cudaEventDestroy(m->tev[i]);
    free(m->tev);
    free(m->twork);
  }
  if (m->own_arena) cudaFree(m->arena);
  free(m);
  return GPT2_OK;
}

static int check_shape(gpt2_t* m, int B, int T) {
  if (B < 1 || T < 1 || B > m->maxB || T > m->maxT || T > m->cfg.max_seq_len) return GPT2_ERR_SHAPE;
  return GPT2_OK;
}

static int read_device_status(gpt2_t* m) {
  int err = 0;
  CCHECK(m, cudaStreamSynchronize(m->stream));
  CCHECK(m, cudaMemcpy(&err, m->err, sizeof(int), cudaMemcpyDeviceToHost));
  if (err == DEV_OK) return GPT2_OK;
  CCHECK(m, cudaMemset(m->err, 0, sizeof(int)));
  if (err == DEV_ERR_TOKEN_RANGE) return GPT2_ERR_TOKEN_RANGE;
  if (err == DEV_ERR_TIMEOUT) {
    m->poisoned = GPT2_ERR_DEVICE_TIMEOUT;
    return GPT2_ERR_DEVICE_TIMEOUT;
  }
  return GPT2_ERR_SHAPE;
}

EXPORT int gpt2_sync(gpt2_t* m, float* loss_out) {
  if (!m) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  int rc = read_device_status(m);
  if (rc != GPT2_OK) return rc;
  if (loss_out) {
    if (!m->have_targets) {
      *loss_out = -1.0f;
      return GPT2_OK;
    }
    CCHECK(m, cudaMemcpy(loss_out, m->loss, sizeof(float), cudaMemcpyDeviceToHost));
    if (!isfinite(*loss_out)) return GPT2_WARN_NONFINITE;
  }
  return GPT2_OK;
}

EXPORT int gpt2_forward(gpt2_t* m, const int32_t* inputs, const int32_t* targets, int B, int T, float* loss_out) {
  if (!m || !inputs) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  int rc = check_shape(m, B, T);
  if (rc) return rc;
  int N = B * T, V = m->cfg.vocab_size;
  for (int i = 0; i < N; i++) {
    if (inputs[i] < 0 || inputs[i] >= V) return GPT2_ERR_TOKEN_RANGE;
    if (targets && (targets[i] < 0 || targets[i] >= V)) return GPT2_ERR_TOKEN_RANGE;
  }
  m->launches = 0;
  CCHECK(m, cudaMemcpyAsync(m->tokens, inputs, N * sizeof(int), cudaMemcpyHostToDevice, m->stream));
  if (targets) CCHECK(m, cudaMemcpyAsync(m->targets, targets, N * sizeof(int), cudaMemcpyHostToDevice, m->stream));
  rc = enqueue_forward(m, m->tokens, targets ? m->targets : nullptr, B, T, 0);
  if (rc) return rc;
  if (loss_out) return gpt2_sync(m, loss_out);
  return GPT2_OK;
}

// Generation (the pages' sample_mult loop): for t = n_prompt .. n_total-1, a
// forward of batch row 0 over all n_total positions, then one draw from the
// softmax of logits row t-1 with coin t - n_prompt, written to position t of
// the device token buffer, where the next forward reads it.  Positions not
// yet sampled hold the first prompt token; causal attention keeps them out of
// the logits that are read.  The coins are staged in the per-row loss buffer,
// which a forward without targets does not use.
EXPORT int gpt2_sample(gpt2_t* m, int32_t* tokens, int n_prompt, int n_total, const float* coins) {
  if (!m || !tokens || !coins) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  if (n_prompt < 1 || n_total <= n_prompt) return GPT2_ERR_ARG;
  int rc = check_shape(m, 1, n_total);
  if (rc) return rc;
  const int V = m->cfg.vocab_size, Vp = m->cfg.padded_vocab_size, ncoins = n_total - n_prompt;
  for (int i = 0; i < n_prompt; i++)
    if (tokens[i] < 0 || tokens[i] >= V) return GPT2_ERR_TOKEN_RANGE;
  for (int i = 0; i < ncoins; i++)
    if (!(coins[i] >= 0.f && coins[i] < 1.f)) return GPT2_ERR_ARG;
  m->launches = 0;
  std::vector<int32_t> init(tokens, tokens + n_total);
  for (int i = n_prompt; i < n_total; i++) init[i] = tokens[0];
  CCHECK(m, cudaMemcpyAsync(m->tokens, init.data(), (size_t)n_total * sizeof(int32_t), cudaMemcpyHostToDevice,
                            m->stream));
  CCHECK(m, cudaMemcpyAsync(m->losses, coins, (size_t)ncoins * sizeof(float), cudaMemcpyHostToDevice, m->stream));
  for (int t = n_prompt; t < n_total; t++) {
    rc = enqueue_forward(m, m->tokens, nullptr, 1, n_total, 0);
    if (rc) return rc;
    launch_k(sample_kernel, 1, SAMPLE_THREADS, 0, m->stream, m->tokens, t, m->logits + (size_t)(t - 1) * Vp, V,
             (const float*)m->losses, t - n_prompt);
    m->launches++;
  }
  CCHECK(m, cudaMemcpyAsync(tokens, m->tokens, (size_t)n_total * sizeof(int32_t), cudaMemcpyDeviceToHost, m->stream));
  return read_device_status(m);
}

EXPORT int gpt2_forward_device(gpt2_t* m, const int32_t* d_inputs, const int32_t* d_targets, int B, int T) {
  if (!m || !d_inputs) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  int rc = check_shape(m, B, T);
  if (rc) return rc;
  int N = B * T;
  m->launches = 0;
  // stage into the handle's buffers: the embedding backward reads the ids later
  if (d_inputs != m->tokens)
    CCHECK(m, cudaMemcpyAsync(m->tokens, d_inputs, N * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
  if (d_targets && d_targets != m->targets)
    CCHECK(m, cudaMemcpyAsync(m->targets, d_targets, N * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
  return enqueue_forward(m, m->tokens, d_targets ? m->targets : nullptr, B, T, 1);
}

EXPORT int gpt2_zero_grad(gpt2_t* m) {
  if (!m) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  m->launches = 0;
  CCHECK(m, cudaMemsetAsync(m->grads, 0, m->np * sizeof(float), m->stream));
  return GPT2_OK;
}

EXPORT int gpt2_backward(gpt2_t* m) {
  if (!m) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  if (!m->fwd_done || !m->have_targets) return GPT2_ERR_STATE;
  m->launches = 0;
  return enqueue_backward(m);
}

EXPORT int gpt2_update(gpt2_t* m, float lr, float beta1, float beta2, float eps, float weight_decay, int t) {
  if (!m || t < 1) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  m->launches = 0;
  int rc = write_hparams(m, lr, beta1, beta2, eps, weight_decay, t);
  return rc ? rc : enqueue_update(m);
}

// forward (device-side token check) -> zero_grad -> backward -> AdamW, all
// reading the staged tokens and the device-resident hyper-parameters.
// forward -> zero_grad -> backward -> update.  zero_grad followed by an
// accumulating backward equals a backward that stores its gradients, so the
// fused step skips the 4*Np-byte clear: every gradient is stored exactly once
// (the LM-head weight gradient first, then the embedding rows added on top),
// except the wpe rows at positions >= T, which are cleared.
static int enqueue_step(gpt2_t* m, int B, int T) {
  int rc;
  if ((rc = enqueue_forward(m, m->tokens, m->targets, B, T, 1))) return rc;
  const int C = m->cfg.channels;
  if (m->cfg.max_seq_len > T && !m->cfg.llama)  // (the Llama-style variant has no position table)
    CCHECK(m, cudaMemsetAsync(m->G[P_WPE] + (size_t)T * C, 0, (size_t)(m->cfg.max_seq_len - T) * C * sizeof(float),
                              m->stream));
  m->grad_accumulate = 0;
  m->upd_layers = 1;  // each layer's AdamW starts once its gradients are complete
  rc = enqueue_backward(m);
  m->upd_layers = 0;
  m->grad_accumulate = 1;
  if (rc) return rc;
  return update_rest(m, B * T);
}

static int run_step(gpt2_t* m, int B, int T, int use_graph) {
  m->launches = 0;
  // the legacy default stream cannot be captured; the timer needs direct launches
  if (!use_graph || m->stream == nullptr || m->timer_kind != TK_NONE) return enqueue_step(m, B, T);
  if (!m->gexec || m->gB != B || m->gT != T) {
    if (m->gexec) {
      cudaGraphExecDestroy(m->gexec);
      m->gexec = nullptr;
    }
    CCHECK(m, cudaStreamBeginCapture(m->stream, cudaStreamCaptureModeThreadLocal));
    m->capturing = 1;
    int rc = enqueue_step(m, B, T);
    m->capturing = 0;
    cudaGraph_t g = nullptr;
    cudaError_t e = cudaStreamEndCapture(m->stream, &g);
    if (rc) {
      if (g) cudaGraphDestroy(g);
      return rc;
    }
    CCHECK(m, e);
    e = cudaGraphInstantiate(&m->gexec, g, 0);
    cudaGraphDestroy(g);
    CCHECK(m, e);
    m->gB = B;
    m->gT = T;
    m->g_launches = m->launches;
  }
  CCHECK(m, cudaGraphLaunch(m->gexec, m->stream));
  m->launches = m->g_launches;
  m->B = B;
  m->T = T;
  m->have_targets = 1;
  m->fwd_done = 1;
  return GPT2_OK;
}

EXPORT int gpt2_train_step_device(gpt2_t* m, const int32_t* d_inputs, const int32_t* d_targets, int B, int T,
                                  float lr, float beta1, float beta2, float eps, float weight_decay, int t,
                                  int use_graph) {
  if (!m || !d_inputs || !d_targets || t < 1) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  int rc = check_shape(m, B, T);
  if (rc) return rc;
  int N = B * T;
  if (d_inputs != m->tokens)
    CCHECK(m, cudaMemcpyAsync(m->tokens, d_inputs, N * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
  if (d_targets != m->targets)
    CCHECK(m, cudaMemcpyAsync(m->targets, d_targets, N * sizeof(int), cudaMemcpyDeviceToDevice, m->stream));
  if ((rc = write_hparams(m, lr, beta1, beta2, eps, weight_decay, t))) return rc;
  return run_step(m, B, T, use_graph);
}

EXPORT int gpt2_train_step(gpt2_t* m, const int32_t* inputs, const int32_t* targets, int B, int T, float lr,
                           float beta1, float beta2, float eps, float weight_decay, int t, float* loss_out) {
  if (!m || !inputs || !targets || t < 1) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  int rc = check_shape(m, B, T);
  if (rc) return rc;
  int N = B * T, V = m->cfg.vocab_size;
  for (int i = 0; i < N; i++)
    if (inputs[i] < 0 || inputs[i] >= V || targets[i] < 0 || targets[i] >= V) return GPT2_ERR_TOKEN_RANGE;
  CCHECK(m, cudaMemcpyAsync(m->tokens, inputs, N * sizeof(int), cudaMemcpyHostToDevice, m->stream));
  CCHECK(m, cudaMemcpyAsync(m->targets, targets, N * sizeof(int), cudaMemcpyHostToDevice, m->stream));
  if ((rc = write_hparams(m, lr, beta1, beta2, eps, weight_decay, t))) return rc;
  if ((rc = run_step(m, B, T, 1))) return rc;
  return gpt2_sync(m, loss_out);
}

EXPORT int gpt2_kernel_timer(gpt2_t* m, int kind) {
  if (!m || kind < 0 || kind > TK_ENCODER) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  if (!m->tev) {
    m->tcap = 4096;
    m->tev = (cudaEvent_t*)calloc(2 * m->tcap, sizeof(cudaEvent_t));
    m->twork = (double*)calloc(m->tcap, sizeof(double));
    for (int i = 0; i < 2 * m->tcap; i++) CCHECK(m, cudaEventCreate(&m->tev[i]));
  }
  timer_drain(m);
  m->timer_kind = kind;
  m->t_ms = 0.0;
  m->t_work = 0.0;
  m->t_launches = 0;
  return GPT2_OK;
}

EXPORT int gpt2_kernel_timer_read(gpt2_t* m, double* total_ms, long long* launches, double* total_work) {
  if (!m || !total_ms || !launches || !total_work) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  timer_drain(m);
  *total_ms = m->t_ms;
  *launches = m->t_launches;
  *total_work = m->t_work;
  return GPT2_OK;
}

EXPORT int gpt2_set_wait_limit_ns(unsigned long long ns) {
  const unsigned long long v = ns ? ns : (unsigned long long)tc::WAIT_LIMIT_NS;
  if (cudaMemcpyToSymbol(tc::g_wait_limit_ns, &v, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return GPT2_ERR_CUDA;
  }
  return cudaDeviceSynchronize() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

EXPORT int gpt2_plan_bf16_matmul(int M, int N, int K, int no_split, int logits, int num_sms, int* BN, int* splits) {
  if (M <= 0 || N <= 0 || K <= 0 || num_sms <= 0 || !BN || !splits) return GPT2_ERR_ARG;
  const Bf16Plan plan = plan_bf16(M, N, K, no_split || logits, SPLITK_WS_FLOATS, num_sms, !logits);
  *BN = plan.BN;
  *splits = plan.splits;
  return GPT2_OK;
}

EXPORT long long gpt2_num_parameters(const gpt2_t* m) { return m ? m->np : -1; }

EXPORT long long gpt2_last_launch_count(const gpt2_t* m) { return m ? m->launches : -1; }

static int copy_flat(gpt2_t* m, void* dst, const void* src, long long n, cudaMemcpyKind kind) {
  if (!m || !dst || !src) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  if (n != m->np) return GPT2_ERR_ARG;
  CCHECK(m, cudaStreamSynchronize(m->stream));
  CCHECK(m, cudaMemcpy(dst, src, n * sizeof(float), kind));
  return GPT2_OK;
}

EXPORT int gpt2_get_params(gpt2_t* m, float* host, long long n) {
  return copy_flat(m, host, m ? m->params : nullptr, n, cudaMemcpyDeviceToHost);
}

EXPORT int gpt2_set_params(gpt2_t* m, const float* host, long long n) {
  int rc = copy_flat(m, m ? m->params : nullptr, host, n, cudaMemcpyHostToDevice);
  if (rc) return rc;
  rc = refresh_bf16(m);
  if (rc) return rc;
  CCHECK(m, cudaStreamSynchronize(m->stream));
  return GPT2_OK;
}

EXPORT int gpt2_get_grads(gpt2_t* m, float* host, long long n) {
  return copy_flat(m, host, m ? m->grads : nullptr, n, cudaMemcpyDeviceToHost);
}

EXPORT int gpt2_get_opt_state(gpt2_t* m, float* hm, float* hv, long long n) {
  int rc = copy_flat(m, hm, m ? m->m : nullptr, n, cudaMemcpyDeviceToHost);
  return rc ? rc : copy_flat(m, hv, m->v, n, cudaMemcpyDeviceToHost);
}

EXPORT int gpt2_set_opt_state(gpt2_t* m, const float* hm, const float* hv, long long n) {
  int rc = copy_flat(m, m ? m->m : nullptr, hm, n, cudaMemcpyHostToDevice);
  return rc ? rc : copy_flat(m, m->v, hv, n, cudaMemcpyHostToDevice);
}

EXPORT int gpt2_get_logits(gpt2_t* m, float* host, long long n) {
  if (!m || !host) return GPT2_ERR_ARG;
  if (m->poisoned) return m->poisoned;
  if (!m->fwd_done) return GPT2_ERR_STATE;
  if (n != (long long)m->B * m->T * m->cfg.padded_vocab_size) return GPT2_ERR_ARG;
  CCHECK(m, cudaStreamSynchronize(m->stream));
  if (!m->logits_in_bf) {
    CCHECK(m, cudaMemcpy(host, m->logits, n * sizeof(float), cudaMemcpyDeviceToHost));
    return GPT2_OK;
  }
  // bf16 logits: widened to fp32 exactly (a bf16 value is the top half of an fp32 one)
  std::vector<uint16_t> tmp((size_t)n);
  CCHECK(m, cudaMemcpy(tmp.data(), m->logits_bf, n * sizeof(uint16_t), cudaMemcpyDeviceToHost));
  for (long long i = 0; i < n; i++) {
    const uint32_t u = (uint32_t)tmp[(size_t)i] << 16;
    memcpy(&host[i], &u, sizeof(float));
  }
  return GPT2_OK;
}

// ---------------------------------------------------------------------------
// kernel-level entry points (device buffers), for per-layer parity tests
// ---------------------------------------------------------------------------
// workspace layout: [error word (256 B)][tile counters][bias partials ceil(N/64) x OC][split-K partials]
// [bf16 copies of x (N x IC), W (OC x IC), dy (N x OC)]
static size_t al256(size_t b) { return (b + 255) & ~(size_t)255; }

EXPORT size_t gpt2op_matmul_workspace_bytes(int N, int IC, int OC) {
  if (N < 1 || IC < 1 || OC < 1) return 0;
  size_t bias = (size_t)ceil_div(N, 64) * OC * sizeof(float);
  return OP_HDR_BYTES + al256(bias) + SPLITK_WS_FLOATS * sizeof(float) + al256((size_t)N * IC * 2) +
         al256((size_t)OC * IC * 2) + al256((size_t)N * OC * 2);
}

struct OpWs {
  int* err;
  int* tile_ctr;
  float* bias_partial;
  float* splitk;
  long long splitk_floats;
  uint16_t *xbf, *Wbf, *dybf;  // bf16 operand copies (bf16 precision)
};

static OpWs op_ws(void* ws, int N, int IC, int OC) {
  OpWs w;
  char* b = (char*)ws;
  size_t bias = al256((size_t)ceil_div(N, 64) * OC * sizeof(float));
  w.err = (int*)b;
  w.tile_ctr = (int*)(b + 256);
  w.bias_partial = (float*)(b + OP_HDR_BYTES);
  w.splitk = (float*)(b + OP_HDR_BYTES + bias);
  w.splitk_floats = SPLITK_WS_FLOATS;
  char* h = b + OP_HDR_BYTES + bias + SPLITK_WS_FLOATS * sizeof(float);
  w.xbf = (uint16_t*)h;
  w.Wbf = (uint16_t*)(h + al256((size_t)N * IC * 2));
  w.dybf = (uint16_t*)(h + al256((size_t)N * IC * 2) + al256((size_t)OC * IC * 2));
  return w;
}

static int op_to_bf16(const float* x, uint16_t* y, long long n, cudaStream_t s) {
  launch_k(to_bf16_kernel, grid_for(n, 256), 256, 0, s, x, y, n);
  return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

static int op_matmul(const MatmulDesc& d, int precision, const OpWs& w, cudaStream_t s) {
  int n = precision == GPT2_PREC_BF16 ? launch_matmul_bf16(d, w.splitk, w.tile_ctr, w.err, s, w.splitk_floats)
                                      : launch_matmul(d, s, w.err);
  if (n < 0) return GPT2_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

static int op_status(const OpWs& w, cudaStream_t s) {
  int err = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return GPT2_ERR_CUDA;
  if (cudaMemcpy(&err, w.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return GPT2_ERR_CUDA;
  if (err == DEV_ERR_TIMEOUT) return GPT2_ERR_DEVICE_TIMEOUT;
  return err ? GPT2_ERR_SHAPE : GPT2_OK;
}

static int op_prepare(void* workspace, cudaStream_t s) {
  if (set_kernel_attributes() != GPT2_OK) return GPT2_ERR_CUDA;
  // clears the error word and the split-K tile counters
  return cudaMemsetAsync(workspace, 0, OP_HDR_BYTES, s) == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

static int op_check_shape(int N, int IC, int OC, int precision) {
  if (precision != GPT2_PREC_FP32 && precision != GPT2_PREC_BF16) return GPT2_ERR_ARG;
  // TMA rows must be multiples of 16 bytes
  int q = precision == GPT2_PREC_BF16 ? 8 : 4;
  if (IC % q || OC % q) return GPT2_ERR_SHAPE;
  return GPT2_OK;
}

EXPORT int gpt2op_matmul_forward(float* out, const float* x, const float* W, const float* bias, int N, int IC, int OC,
                                 int precision, void* workspace, void* stream) {
  if (!out || !x || !W || !workspace || N < 1 || IC < 1 || OC < 1) return GPT2_ERR_ARG;
  int rc = op_check_shape(N, IC, OC, precision);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if ((rc = op_prepare(workspace, s))) return rc;
  OpWs w = op_ws(workspace, N, IC, OC);
  if (precision == GPT2_PREC_BF16) {
    if ((rc = op_to_bf16(x, w.xbf, (long long)N * IC, s)) || (rc = op_to_bf16(W, w.Wbf, (long long)OC * IC, s)))
      return rc;
  }
  MatmulDesc d = {N, OC, IC, x, IC, 1, W, IC, 1, epi_args(out, OC, bias ? EPI_BIAS : EPI_STORE, bias), w.xbf, w.Wbf};
  rc = op_matmul(d, precision, w, s);
  return rc ? rc : op_status(w, s);
}

static int op_backward(float* dx, float* dW, float* dbias, const float* dy, const float* x, const float* W, int N,
                       int IC, int OC, int precision, const OpWs& w, cudaStream_t s) {
  int rc;
  if (precision == GPT2_PREC_BF16) {
    if ((rc = op_to_bf16(x, w.xbf, (long long)N * IC, s)) || (rc = op_to_bf16(W, w.Wbf, (long long)OC * IC, s)) ||
        (rc = op_to_bf16(dy, w.dybf, (long long)N * OC, s)))
      return rc;
  }
  MatmulDesc ddx = {N, IC, OC, dy, OC, 1, W, IC, 0, epi_args(dx, IC, EPI_STORE), w.dybf, w.Wbf};
  if ((rc = op_matmul(ddx, precision, w, s))) return rc;
  MatmulDesc ddw = {OC, IC, N, dy, OC, 0, x, IC, 0, epi_args(dW, IC, EPI_ACCUM), w.dybf, w.xbf};
  if ((rc = op_matmul(ddw, precision, w, s))) return rc;
  if (dbias) {
    // 64-row chunks, doubled while the chunks would exceed the grid's y limit:
    // never more partial rows than ceil(N/64), which the scratch is sized for
    int rows = 64;
    while (ceil_div(N, rows) > 65535) rows *= 2;
    const int chunks = ceil_div(N, rows);
    launch_k(col_partial_kernel, dim3(ceil_div(OC, 256), chunks), 256, 0, s, dy, N, OC, OC, rows, w.bias_partial);
    launch_k(col_finish_kernel, ceil_div(OC, 32), COLF_WARPS * 32, 0, s, dbias, dbias, dbias, OC, w.bias_partial,
             chunks, OC, 1);
    if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
  }
  return op_status(w, s);
}

EXPORT int gpt2op_matmul_backward(float* dx, float* dW, float* dbias, const float* dy, const float* x, const float* W,
                                  int N, int IC, int OC, int precision, void* workspace, void* stream) {
  if (!dx || !dW || !dy || !x || !W || !workspace || N < 1 || IC < 1 || OC < 1) return GPT2_ERR_ARG;
  int rc = op_check_shape(N, IC, OC, precision);
  if (rc) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if ((rc = op_prepare(workspace, s))) return rc;
  return op_backward(dx, dW, dbias, dy, x, W, N, IC, OC, precision, op_ws(workspace, N, IC, OC), s);
}

// attention forward: workspace = [error word, 256 B][bf16 copy of qkv]
EXPORT size_t gpt2op_attention_workspace_bytes(int B, int T, int C) {
  if (B < 1 || T < 1 || C < 1) return 0;
  return 256 + al256((size_t)B * T * 3 * C * 2);
}

EXPORT int gpt2op_attention_forward(float* y, float* lse, const float* qkv, int B, int T, int C, int NH, int precision,
                                    void* workspace, void* stream) {
  if (!y || !lse || !qkv || !workspace || B < 1 || T < 1 || C < 1 || NH < 1) return GPT2_ERR_ARG;
  if (precision != GPT2_PREC_FP32 && precision != GPT2_PREC_BF16) return GPT2_ERR_ARG;
  if (C % NH || C / NH > 128 || C % 8) return GPT2_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  if (set_kernel_attributes() != GPT2_OK) return GPT2_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return GPT2_ERR_CUDA;
  OpWs w = {};
  w.err = (int*)workspace;
  uint16_t* qkv_bf = (uint16_t*)((char*)workspace + 256);
  const int bf = precision == GPT2_PREC_BF16;
  if (bf && op_to_bf16(qkv, qkv_bf, (long long)B * T * 3 * C, s)) return GPT2_ERR_CUDA;
  if (launch_attn_fwd(y, nullptr, lse, qkv, bf ? qkv_bf : nullptr, B, T, C, NH, bf, w.err, s) < 0) return GPT2_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
  return op_status(w, s);
}

// attention backward: workspace = [error word][bf16 qkv][bf16 dy][y][lse][D, or (-lse log2 e, -D) pairs]
EXPORT size_t gpt2op_attention_backward_workspace_bytes(int B, int T, int C, int NH) {
  if (B < 1 || T < 1 || C < 1 || NH < 1) return 0;
  size_t n = (size_t)B * T;
  return 256 + al256(n * 3 * C * 2) + al256(n * C * 2) + al256(n * C * 4) + al256(n * NH * 4) + al256(n * NH * 8);
}

EXPORT int gpt2op_attention_backward(float* dqkv, const float* dy, const float* qkv, int B, int T, int C, int NH,
                                     int precision, void* workspace, void* stream) {
  if (!dqkv || !dy || !qkv || !workspace || B < 1 || T < 1 || C < 1 || NH < 1) return GPT2_ERR_ARG;
  if (precision != GPT2_PREC_FP32 && precision != GPT2_PREC_BF16) return GPT2_ERR_ARG;
  if (C % NH || C / NH > 128 || C % 8) return GPT2_ERR_SHAPE;
  cudaStream_t s = (cudaStream_t)stream;
  if (set_kernel_attributes() != GPT2_OK) return GPT2_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, 256, s) != cudaSuccess) return GPT2_ERR_CUDA;
  size_t n = (size_t)B * T;
  char* w = (char*)workspace;
  OpWs ws = {};
  ws.err = (int*)w;
  uint16_t* qkv_bf = (uint16_t*)(w + 256);
  uint16_t* dy_bf = (uint16_t*)((char*)qkv_bf + al256(n * 3 * C * 2));
  float* y = (float*)((char*)dy_bf + al256(n * C * 2));
  float* lse = (float*)((char*)y + al256(n * C * 4));
  float* D = (float*)((char*)lse + al256(n * NH * 4));
  const int bf = precision == GPT2_PREC_BF16;
  if (bf && (op_to_bf16(qkv, qkv_bf, (long long)n * 3 * C, s) || op_to_bf16(dy, dy_bf, (long long)n * C, s)))
    return GPT2_ERR_CUDA;
  if (launch_attn_fwd(y, nullptr, lse, qkv, bf ? qkv_bf : nullptr, B, T, C, NH, bf, ws.err, s) < 0) return GPT2_ERR_CUDA;
  if (launch_attn_bwd(dqkv, nullptr, D, dy, bf ? dy_bf : nullptr, qkv, bf ? qkv_bf : nullptr, y, lse, B, T, C, NH, bf,
                      ws.err, s) < 0)
    return GPT2_ERR_CUDA;
  if (cudaGetLastError() != cudaSuccess) return GPT2_ERR_CUDA;
  return op_status(ws, s);
}

// ---------------------------------------------------------------------------
// matmul backward with library-owned scratch (no allocation by anyone)
// ---------------------------------------------------------------------------
// The scratch of gpt2op_matmul_backward (error word, split-K tile counters,
// column-sum partials of the bias gradient) is taken from one fixed array in
// the library's device memory.  Every GPU that loads the library holds it
// until the process exits.  Layout: [error word, 256 B][tile counters]
// [column-sum partials, NOALLOC_BIAS_FLOATS floats].  The fp32 matmul reduces
// its K splits inside a thread-block cluster, so it needs no split-K partials.
#define NOALLOC_BIAS_FLOATS ((long long)1 << 21)
#define NOALLOC_SCRATCH_BYTES ((size_t)OP_HDR_BYTES + (size_t)NOALLOC_BIAS_FLOATS * sizeof(float))
#define NOALLOC_MAX_DEVICES 64

static __device__ __align__(256) unsigned char g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// In host code g_noalloc_scratch names a host-side stand-in, not the device
// array, so the device address is looked up once per device (with that
// device current) and cached.
static void* g_noalloc_addr[NOALLOC_MAX_DEVICES];
static std::mutex g_noalloc_mu;

static int noalloc_scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= NOALLOC_MAX_DEVICES) {
    cudaGetLastError();
    return GPT2_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p) {
      fprintf(stderr, "gpt2b300: cudaGetSymbolAddress(scratch) failed on device %d: %s\n", dev,
              cudaGetErrorString(e));
      cudaGetLastError();
      return GPT2_ERR_CUDA;
    }
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return GPT2_OK;
}

EXPORT int gpt2op_matmul_backward_noalloc(float* dx, float* dW, float* dbias, const float* dy, const float* x,
                                          const float* W, int N, int IC, int OC, int precision, void* stream) {
  if (!dx || !dW || !dy || !x || !W || N < 1 || IC < 1 || OC < 1) return GPT2_ERR_ARG;
  // bf16 operand copies would need scratch that scales with the inputs
  if (precision != GPT2_PREC_FP32) return GPT2_ERR_ARG;
  int rc = op_check_shape(N, IC, OC, precision);
  if (rc) return rc;
  if (dbias && (long long)ceil_div(N, 64) * OC > NOALLOC_BIAS_FLOATS) {
    fprintf(stderr, "gpt2b300: gpt2op_matmul_backward_noalloc: ceil(N/64)*OC = %lld exceeds the fixed scratch "
            "(%lld floats)\n", (long long)ceil_div(N, 64) * OC, NOALLOC_BIAS_FLOATS);
    return GPT2_ERR_SHAPE;
  }
  void* base = nullptr;
  if ((rc = noalloc_scratch_address(&base))) return rc;
  cudaStream_t s = (cudaStream_t)stream;
  if ((rc = op_prepare(base, s))) return rc;  // clears the error word and the tile counters
  OpWs w = {};
  w.err = (int*)base;
  w.tile_ctr = (int*)((char*)base + 256);
  w.bias_partial = (float*)((char*)base + OP_HDR_BYTES);
  w.splitk = nullptr;  // read only by the bf16 kernel
  w.splitk_floats = 0;
  return op_backward(dx, dW, dbias, dy, x, W, N, IC, OC, precision, w, s);
}
