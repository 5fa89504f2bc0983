// k_misc.cuh -- parameter init, token validation, embedding forward and
// backward, AdamW, and deterministic column / scalar reductions.
#pragma once
#include "common.cuh"

// ---------------------------------------------------------------------------
// Parameter init: SplitMix64 (Vigna) draw i of stream `seed` is
// mix(seed + (i+1) * golden_gamma); uniforms take the top 53 bits; normal i
// is Box-Muller on the uniform pair (2j, 2j+1), j = i/2, cosine branch for
// even i and sine branch for odd i.
// ---------------------------------------------------------------------------
GPT2_DEV uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
  uint64_t z = seed + (i + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

GPT2_DEV double uniform53_at(uint64_t seed, uint64_t i) {
  return (double)(splitmix64_at(seed, i) >> 11) * 0x1p-53;
}

GPT2_DEV double normal_at(uint64_t seed, uint64_t i) {
  uint64_t j = i >> 1;
  double u0 = uniform53_at(seed, 2 * j), u1 = uniform53_at(seed, 2 * j + 1);
  double r = sqrt(-2.0 * log1p(-u0));
  double a = (2.0 * 3.141592653589793) * u1;
  return (i & 1) ? r * sin(a) : r * cos(a);
}

// Fills p[0 .. n) of the flat buffer that starts at flat offset `base`:
// elements [0, nrand) get std * normal(base + i), the rest `fill`.
__global__ void init_tensor_kernel(float* p, long long base, long long n, long long nrand, double stdv, float fill,
                                   uint64_t seed) {
  pdl_launch_dependents();
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    p[i] = i < nrand ? (float)(stdv * normal_at(seed, (uint64_t)(base + i))) : fill;
}

// ---------------------------------------------------------------------------
// Token ids must lie in [0, V).
// ---------------------------------------------------------------------------
__global__ void validate_tokens_kernel(const int* ids, const int* tgt, int n, int V, int* err) {
  pdl_launch_dependents();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    int a = ids[i];
    int b = tgt ? tgt[i] : 0;
    if (a < 0 || a >= V || b < 0 || b >= V) dev_set_error(err, DEV_ERR_TOKEN_RANGE);
  }
}

// ---------------------------------------------------------------------------
// Token + position embedding: x[b,t,:] = wte[id,:] + wpe[t,:].  One thread
// per float4; C % 4 == 0.  Ids are clamped so that a bad id (already flagged
// by validate_tokens_kernel) cannot read out of bounds.
// ---------------------------------------------------------------------------
__global__ void encoder_fwd_kernel(float* __restrict__ x, const int* __restrict__ ids, const float* __restrict__ wte,
                                   const float* __restrict__ wpe, int BT, int T, int C, int V) {
  pdl_launch_dependents();
  pdl_wait();
  int C4 = C >> 2;
  long long total = (long long)BT * C4;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total; i += (long long)gridDim.x * blockDim.x) {
    int bt = (int)(i / C4), c4 = (int)(i % C4);
    int id = min(max(ids[bt], 0), V - 1);
    int t = bt % T;
    float4 e = reinterpret_cast<const float4*>(wte + (size_t)id * C)[c4];
    // wpe == NULL: no learned position table (the Llama-style variant)
    float4 p = wpe ? reinterpret_cast<const float4*>(wpe + (size_t)t * C)[c4] : make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(x + (size_t)bt * C)[c4] = make_float4(e.x + p.x, e.y + p.y, e.z + p.z, e.w + p.w);
  }
}

// ---------------------------------------------------------------------------
// Embedding backward, deterministic under skewed token frequencies.
//  1. Sort the positions 0..n-1 by (token id, position): sorted[i] is the
//     i-th position of that order, so the positions of one id form a run, in
//     increasing order.  Up to SORT_BITONIC_MAX positions one CTA bitonic-sorts the
//     keys (id << 14 | pos) in shared memory (sort_tokens_kernel); beyond it a
//     stable least-significant-digit radix sort by the id, two passes of 8
//     bits (radix_hist_kernel, radix_scan_kernel, radix_scatter_kernel).
//  2. run_starts_kernel lists where each id's run starts; wte_grad_kernel
//     sums each run's gradient rows in a fixed order and adds the sum to
//     dwte[id] once.
//  3. wpe_grad_kernel: dwpe[t] += sum over b of dx[b,t].
// Limits: V <= 65536.
// ---------------------------------------------------------------------------
#define SORT_MAX 16384         // the bitonic sort's capacity (its keys hold 14 position bits)
#define SORT_BITONIC_MAX 2048  // up to this many positions the bitonic sort (one launch) is the faster

__global__ void __launch_bounds__(1024) sort_tokens_kernel(const int* __restrict__ ids, int n, int V,
                                                          uint32_t* __restrict__ sorted) {
  pdl_launch_dependents();
  pdl_wait();
  extern __shared__ uint32_t keys[];
  int P = 1;
  while (P < n) P <<= 1;
  for (int i = threadIdx.x; i < P; i += blockDim.x) {
    uint32_t id = i < n ? (uint32_t)min(max(ids[i], 0), V - 1) : 0xFFFFu;
    keys[i] = i < n ? ((id << 14) | (uint32_t)i) : 0xFFFFFFFFu;
  }
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += blockDim.x) {
        int l = i ^ j;
        if (l > i) {
          uint32_t a = keys[i], b = keys[l];
          bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[l] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < n; i += blockDim.x) sorted[i] = keys[i] & 0x3FFFu;  // the position
}

// ---- stable radix sort of positions by token id (n > SORT_BITONIC_MAX) ----
// A pass sorts by digit (id >> shift) & 255 of the positions src[0..n)
// (identity when src == NULL), keeping the order of equal digits.  Chunks of
// RADIX_CHUNK positions: radix_hist_kernel counts each chunk's digits into
// hist[digit * nchunks + chunk]; radix_scan_kernel turns that table, in that
// (digit-major) order, into exclusive offsets; radix_scatter_kernel walks
// its chunk in rounds of 256 positions (position order), ranking each
// position among the equal digits before it (warp match, then warp counts in
// warp order, then the counts of earlier rounds), and writes it to
// dst[offset + rank].  Every count is an integer, so the result does not
// depend on execution order.
#define RADIX_THREADS 256
#define RADIX_ROUNDS 16
#define RADIX_CHUNK (RADIX_THREADS * RADIX_ROUNDS)

GPT2_DEV uint32_t radix_digit(const int* ids, int V, uint32_t pos, int shift) {
  return ((uint32_t)min(max(ids[pos], 0), V - 1) >> shift) & 255u;
}

__global__ void __launch_bounds__(RADIX_THREADS) radix_hist_kernel(const int* __restrict__ ids, int V,
                                                                    const uint32_t* __restrict__ src, int n, int shift,
                                                                    int* __restrict__ hist) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int cnt[256];
  cnt[threadIdx.x] = 0;
  __syncthreads();
  const int c0 = blockIdx.x * RADIX_CHUNK;
  for (int i = c0 + threadIdx.x; i < min(n, c0 + RADIX_CHUNK); i += RADIX_THREADS)
    atomicAdd(&cnt[radix_digit(ids, V, src ? src[i] : (uint32_t)i, shift)], 1);
  __syncthreads();
  hist[threadIdx.x * gridDim.x + blockIdx.x] = cnt[threadIdx.x];
}

// One CTA: exclusive prefix sum of hist[0..len) in index order.
__global__ void __launch_bounds__(1024) radix_scan_kernel(int* __restrict__ hist, int len) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int part[1024];
  const int per = (len + 1023) / 1024, i0 = threadIdx.x * per, i1 = min(len, i0 + per);
  int s = 0;
  for (int i = i0; i < i1; i++) s += hist[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // inclusive scan of the per-thread sums
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = threadIdx.x ? part[threadIdx.x - 1] : 0;
  for (int i = i0; i < i1; i++) {
    const int c = hist[i];
    hist[i] = run;
    run += c;
  }
}

__global__ void __launch_bounds__(RADIX_THREADS) radix_scatter_kernel(const int* __restrict__ ids, int V,
                                                                       const uint32_t* __restrict__ src, int n,
                                                                       int shift, const int* __restrict__ offs,
                                                                       uint32_t* __restrict__ dst) {
  pdl_launch_dependents();
  pdl_wait();
  constexpr int W = RADIX_THREADS / 32;
  __shared__ int run[256];     // positions of each digit placed by earlier rounds
  __shared__ int wcnt[W][256]; // this round's count of each digit per warp
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  run[threadIdx.x] = offs[threadIdx.x * gridDim.x + blockIdx.x];
  const int c0 = blockIdx.x * RADIX_CHUNK;
  for (int r = 0; r < RADIX_ROUNDS; r++) {
    const int i = c0 + r * RADIX_THREADS + threadIdx.x;
    const bool live = i < n;
    const uint32_t pos = live ? (src ? src[i] : (uint32_t)i) : 0u;
    const uint32_t d = live ? radix_digit(ids, V, pos, shift) : 256u;  // 256: no digit
    const unsigned peers = __match_any_sync(0xffffffffu, d);
    const int before = __popc(peers & ((1u << lane) - 1u));
    for (int k = threadIdx.x; k < W * 256; k += RADIX_THREADS) (&wcnt[0][0])[k] = 0;
    __syncthreads();
    if (live && before == 0) wcnt[warp][d] = __popc(peers);  // the warp's count of d, by its first lane
    __syncthreads();
    if (live) {
      int rank = run[d] + before;
      for (int w = 0; w < warp; w++) rank += wcnt[w][d];
      dst[rank] = pos;
    }
    __syncthreads();
    {  // digit threadIdx.x: add this round's counts
      int add = 0;
      for (int w = 0; w < W; w++) add += wcnt[w][threadIdx.x];
      run[threadIdx.x] += add;
    }
    __syncthreads();
  }
}

// The runs of the sorted positions: runs[k] = the first index i of the k-th
// run of equal ids (i == 0 or id(sorted[i]) != id(sorted[i-1])), in order;
// *count = the number of runs.  One CTA: thread t scans the contiguous slice
// [t per, (t+1) per), the slices' counts are scanned in thread order.
__global__ void __launch_bounds__(1024) run_starts_kernel(const uint32_t* __restrict__ sorted,
                                                          const int* __restrict__ ids, int V, int n,
                                                          int* __restrict__ runs, int* __restrict__ count) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int part[1024];
  const int per = (n + 1023) / 1024, i0 = threadIdx.x * per, i1 = min(n, i0 + per);
  auto id_at = [&](int i) { return min(max(ids[sorted[i]], 0), V - 1); };
  int c = 0;
  for (int i = i0; i < i1; i++) c += (i == 0 || id_at(i) != id_at(i - 1)) ? 1 : 0;
  part[threadIdx.x] = c;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {
    const int v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int k = threadIdx.x ? part[threadIdx.x - 1] : 0;
  for (int i = i0; i < i1; i++)
    if (i == 0 || id_at(i) != id_at(i - 1)) runs[k++] = i;
  if (threadIdx.x == 1023) *count = part[1023];
}

// grid: (G, ceil(C/128)); block: WTE_WARPS warps; lane l owns channels
// 4*(blockIdx.y*32 + l) .. +3.  CTA x walks the runs x, x + G, ...; for a run
// (one id's positions, from runs[k] up to runs[k+1] or n), warp w sums the
// run's rows w, w + WTE_WARPS, ... in order and the warp sums are added in
// warp order: a fixed summation order for any run length.
#define WTE_WARPS 8
__global__ void __launch_bounds__(WTE_WARPS * 32) wte_grad_kernel(float* __restrict__ dwte, const float* __restrict__ dx,
                                                                  const uint32_t* __restrict__ sorted,
                                                                  const int* __restrict__ ids, int V,
                                                                  const int* __restrict__ runs,
                                                                  const int* __restrict__ nruns, int n, int C) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float4 s_part[WTE_WARPS][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = (blockIdx.y * 32 + lane) * 4;
  const int count = *nruns;
  for (int k = blockIdx.x; k < count; k += gridDim.x) {
    const int i = runs[k], end = k + 1 < count ? runs[k + 1] : n;
    const int id = min(max(ids[sorted[i]], 0), V - 1);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c < C) {
#pragma unroll 4
      for (int j = i + warp; j < end; j += WTE_WARPS) {
        const int pos = (int)sorted[j];
        const float4 g = *reinterpret_cast<const float4*>(dx + (size_t)pos * C + c);
        acc.x += g.x; acc.y += g.y; acc.z += g.z; acc.w += g.w;
      }
    }
    s_part[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c < C) {
      float4 t = s_part[0][lane];
#pragma unroll
      for (int w = 1; w < WTE_WARPS; w++) {
        const float4 u = s_part[w][lane];
        t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
      }
      float4* d = reinterpret_cast<float4*>(dwte + (size_t)id * C + c);
      const float4 o = *d;
      *d = make_float4(o.x + t.x, o.y + t.y, o.z + t.z, o.w + t.w);
    }
    __syncthreads();
  }
}

// accumulate = 0 stores the sums instead of adding them (the fused training
// step, whose gradients start from zero).
__global__ void wpe_grad_kernel(float* __restrict__ dwpe, const float* __restrict__ dx, int B, int T, int C,
                                int accumulate) {
  pdl_launch_dependents();
  pdl_wait();
  int C4 = C >> 2;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < T * C4; i += gridDim.x * blockDim.x) {
    int t = i / C4, c4 = i % C4;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b = 0; b < B; b++) {
      float4 g = reinterpret_cast<const float4*>(dx + ((size_t)b * T + t) * C)[c4];
      s.x += g.x; s.y += g.y; s.z += g.z; s.w += g.w;
    }
    float4* d = reinterpret_cast<float4*>(dwpe + (size_t)t * C) + c4;
    if (accumulate) {
      float4 o = *d;
      s = make_float4(o.x + s.x, o.y + s.y, o.z + s.z, o.w + s.w);
    }
    *d = s;
  }
}

// ---------------------------------------------------------------------------
// Deterministic column sums of a (M, N) row-major matrix, in two stages:
// partial[chunk][col] over row chunks of `rows` rows, then out[col] += the
// chunk partials summed in chunk order.
// ---------------------------------------------------------------------------
__global__ void col_partial_kernel(const float* __restrict__ Y, int M, int N, long long ldy, int rows,
                                   float* __restrict__ partial) {
  pdl_launch_dependents();
  pdl_wait();
  int col = blockIdx.x * blockDim.x + threadIdx.x;
  if (col >= N) return;
  int r0 = blockIdx.y * rows, r1 = min(M, r0 + rows);
  float s = 0.f;
#pragma unroll 8
  for (int r = r0; r < r1; r++) s += Y[(size_t)r * ldy + col];
  partial[(size_t)blockIdx.y * N + col] = s;
}

// Column sums of partial rows, finished in a fixed order:
//   out[c] += sum_{r < nrows} partial[r][c]   for c < split   (out0)
//   out1[c - split] += ...                    for split <= c < 2 split
//   out2[c - 2 split] += ...                  for c >= 2 split
// (= instead of += when accumulate == 0).  One CTA of 32 warps per 32
// columns: warp w sums rows w, w+32, ... (lane = column, coalesced), then the
// 32 warp sums are added in warp order.
#define COLF_WARPS 32
__global__ void __launch_bounds__(COLF_WARPS * 32) col_finish_kernel(float* __restrict__ out0, float* __restrict__ out1,
                                                                     float* __restrict__ out2, int split,
                                                                     const float* __restrict__ partial, int nrows,
                                                                     int ncols, int accumulate) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float sh[COLF_WARPS][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (c < ncols) {
#pragma unroll 4
    for (int r = warp; r < nrows; r += COLF_WARPS) s += partial[(size_t)r * ncols + c];
  }
  sh[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && c < ncols) {
    float t = sh[0][lane];
#pragma unroll
    for (int w = 1; w < COLF_WARPS; w++) t += sh[w][lane];
    float* o = c < split ? out0 + c : c < 2 * split ? out1 + (c - split) : out2 + (c - 2 * split);
    *o = accumulate ? *o + t : t;
  }
}

// Mean of n values in a fixed order (one CTA of 1024 threads).
__global__ void __launch_bounds__(1024) mean_kernel(const float* __restrict__ x, int n, float* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float sh[32];
  float s = 0.f;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s += x[i];
  s = warp_sum(s);
  if ((threadIdx.x & 31) == 0) sh[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? sh[threadIdx.x] : 0.f;
    v = warp_sum(v);
    if (threadIdx.x == 0) out[0] = v / (float)n;
  }
}

// ---------------------------------------------------------------------------
// AdamW over segments of the flat buffers (float4 granularity).  Segment k
// covers float4 elements [off4[k], off4[k] + (end4[k] - end4[k-1])), end4 the
// running total (end4[-1] = 0); one launch updates one segment list, e.g. the
// whole buffer or the twelve tensors of one layer.  hp holds {lr, beta1,
// beta2, eps, weight_decay, 1/(1-beta1^t), 1/(1-beta2^t)}.  When pbf16 !=
// NULL the bf16 copy of the updated parameters is written too.
// ---------------------------------------------------------------------------
#define ADAMW_MAX_SEGS 16
struct AdamSegs {
  long long off4[ADAMW_MAX_SEGS];
  long long end4[ADAMW_MAX_SEGS];
  int n;
};

// One float4 of AdamW at float4 index i.
GPT2_DEV void adamw_f4(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                       float* __restrict__ v, long long i, const float* __restrict__ hp, uint16_t* __restrict__ pbf16) {
  const float lr = hp[0], b1 = hp[1], b2 = hp[2], eps = hp[3], wd = hp[4], c1inv = hp[5], c2inv = hp[6];
  float4 pp = reinterpret_cast<float4*>(p)[i];
  float4 gg = reinterpret_cast<const float4*>(g)[i];
  float4 mm = reinterpret_cast<float4*>(m)[i];
  float4 vv = reinterpret_cast<float4*>(v)[i];
  float* P = &pp.x;
  const float* G = &gg.x;
  float* Mm = &mm.x;
  float* Vv = &vv.x;
#pragma unroll
  for (int k = 0; k < 4; k++) {
    Mm[k] = b1 * Mm[k] + (1.0f - b1) * G[k];
    Vv[k] = b2 * Vv[k] + (1.0f - b2) * G[k] * G[k];
    float mh = Mm[k] * c1inv, vh = Vv[k] * c2inv;
    P[k] = P[k] - lr * (mh / (sqrtf(vh) + eps) + wd * P[k]);
  }
  reinterpret_cast<float4*>(p)[i] = pp;
  reinterpret_cast<float4*>(m)[i] = mm;
  reinterpret_cast<float4*>(v)[i] = vv;
  if (pbf16) reinterpret_cast<uint2*>(pbf16)[i] = make_uint2(bf16x2_bits(pp.x, pp.y), bf16x2_bits(pp.z, pp.w));
}

__global__ void adamw_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                             float* __restrict__ v, const __grid_constant__ AdamSegs segs,
                             const float* __restrict__ hp, uint16_t* __restrict__ pbf16) {
  pdl_launch_dependents();
  pdl_wait();
  const long long total = segs.end4[segs.n - 1];
  int sg = 0;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    while (e >= segs.end4[sg]) sg++;  // e only grows
    adamw_f4(p, g, m, v, segs.off4[sg] + e - (sg ? segs.end4[sg - 1] : 0), hp, pbf16);
  }
}

// AdamW of the rows r < nrows of a row-major (nrows, C) tensor at element
// offset off whose mask byte mask[r] equals want (C % 4 == 0, off % 4 == 0).
__global__ void adamw_rows_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                                  float* __restrict__ v, long long off, int nrows, int C,
                                  const uint8_t* __restrict__ mask, int want, const float* __restrict__ hp,
                                  uint16_t* __restrict__ pbf16) {
  pdl_launch_dependents();
  pdl_wait();
  const int C4 = C >> 2;
  const long long total = (long long)nrows * C4;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total; e += (long long)gridDim.x * blockDim.x) {
    if (mask[e / C4] != want) continue;
    adamw_f4(p, g, m, v, off / 4 + e, hp, pbf16);
  }
}

// AdamW of the rows of a (rows, C) tensor at element offset off that the
// batch's tokens name: the ids of the runs of the embedding backward's sorted
// positions.  CTA x updates the rows of runs x, x + gridDim.x, ...
__global__ void adamw_sorted_rows_kernel(float* __restrict__ p, const float* __restrict__ g, float* __restrict__ m,
                                         float* __restrict__ v, long long off, int C,
                                         const uint32_t* __restrict__ sorted, const int* __restrict__ ids, int V,
                                         const int* __restrict__ runs, const int* __restrict__ nruns,
                                         const float* __restrict__ hp, uint16_t* __restrict__ pbf16) {
  pdl_launch_dependents();
  pdl_wait();
  const int C4 = C >> 2, count = *nruns;
  for (int k = blockIdx.x; k < count; k += gridDim.x) {
    const int id = min(max(ids[sorted[runs[k]]], 0), V - 1);
    for (int c4 = threadIdx.x; c4 < C4; c4 += blockDim.x) adamw_f4(p, g, m, v, off / 4 + (long long)id * C4 + c4, hp, pbf16);
  }
}

// mask[ids[i]] = 1 for every i < n (the rows of wte a batch touches)
__global__ void mark_rows_kernel(const int* __restrict__ ids, int n, int V, uint8_t* __restrict__ mask) {
  pdl_launch_dependents();
  pdl_wait();
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    mask[min(max(ids[i], 0), V - 1)] = 1;
}

__global__ void to_bf16_kernel(const float* __restrict__ x, uint16_t* __restrict__ y, long long n) {
  pdl_launch_dependents();
  pdl_wait();
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
    y[i] = to_bf16_bits(x[i]);
}
