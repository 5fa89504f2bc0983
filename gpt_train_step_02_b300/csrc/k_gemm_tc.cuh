// k_gemm_tc.cuh -- fp32-accurate matmul on the 5th-generation tensor cores
// (tcgen05.mma kind::tf32, accumulator in TMEM), fed by TMA.
//
//   acc(i,j) = sum_k A(i,k) B(j,k),  i < M, j < N, k < K,
// where each operand is stored either K-major (row i holds its K values
// contiguously) or MN-major (row k holds the M or N values contiguously).
// The three products of a linear layer map onto it as
//   forward          A = x  (K-major), B = W   (K-major)
//   input gradient   A = dy (K-major), B = W   (MN-major)
//   weight gradient  A = dy (MN-major), B = x  (MN-major).
//
// fp32 accuracy with TF32 tensor cores ("3xTF32", the split-precision
// scheme of Ootomo & Yokota, 2022): every operand value is split as
// x = hi + lo with hi = x rounded to TF32 and lo = x - hi (exact), and
// a*b ~ ah*bh + ah*bl + al*bh, three MMAs into one fp32 accumulator.  The
// dropped al*bl term and the TF32 rounding of lo are ~2^-20 relative.
//
// CTA = one 128 x 128 output tile over a range of K, 10 warps.  When K is
// split, the S splits of a tile form one thread-block cluster and are summed
// through distributed shared memory (below).
//   warp 0      one lane issues the TMA loads of raw fp32 tiles (raw ring)
//   warp 1      allocates TMEM; one lane issues tcgen05.mma and commits
//   warps 2..9  split each raw tile into hi/lo halves: A's go to tensor
//               memory (row i in TMEM lane i, one K value per column), B's
//               to shared memory laid out K-major with the 128-byte swizzle
//               (MN-major tiles are transposed on the way); then they run
//               the epilogue: tcgen05.ld TMEM -> registers -> global (two
//               warps per TMEM lane quadrant, 64 columns each).
// The MMAs read A from tensor memory and only B from shared memory, so a K
// tile costs the splitters' raw reads and B writes plus three B reads: about
// half the shared-memory traffic of staging both operands there, which is
// what bounds the main loop.
// Every mbarrier wait is bounded; on expiry the CTA records DEV_ERR_TIMEOUT
// in the error word, stops issuing work, frees its TMEM and returns.
#pragma once
#include <cuda.h>

#include "common.cuh"
#include "gemm_common.cuh"

namespace tc {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 32;  // fp32 elements = 128 bytes: one swizzle row
constexpr int RAW_STAGES = 4;
constexpr int COMP_STAGES = 2;
constexpr int TILE_BYTES = BM * BK * 4;  // 16 KB (A or B tile)
constexpr int SPLIT_WARPS = 8;           // splitter / epilogue warps (two per TMEM lane quadrant)
constexpr int SPLIT_THREADS = 32 * SPLIT_WARPS;
constexpr int THREADS = 64 + SPLIT_THREADS;
// TMEM columns: the 128 x 128 fp32 accumulator in 0..127, then per hi/lo
// stage c the A halves: hi at TM_A + 64c, lo at TM_A + 64c + 32.
constexpr int TM_A = 128;
constexpr int TMEM_COLS = 256;
static_assert(TM_A + COMP_STAGES * 2 * BK <= TMEM_COLS, "A stages must fit the TMEM allocation");
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;  // 1 s of wall time per wait before giving up

// The limit of the pipeline waits (mbar_wait), per device: WAIT_LIMIT_NS
// unless a test lowers it to make them give up (gpt2_set_wait_limit_ns).  The
// drain waits of the abort path always allow WAIT_LIMIT_NS.
__constant__ unsigned long long g_wait_limit_ns = WAIT_LIMIT_NS;

// shared memory map (offsets from a 1024-byte aligned base)
constexpr int OFF_RAW_A = 0;
constexpr int OFF_RAW_B = OFF_RAW_A + RAW_STAGES * TILE_BYTES;
constexpr int OFF_HI_B = OFF_RAW_B + RAW_STAGES * TILE_BYTES;
constexpr int OFF_LO_B = OFF_HI_B + COMP_STAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_LO_B + COMP_STAGES * TILE_BYTES;
// after the main loop (every raw tile consumed) the raw ring holds this CTA's
// split-K partial tile or the epilogue's staging
constexpr int OFF_STAGE = OFF_RAW_A;
constexpr int STAGE_PITCH = BN + 4;  // floats per staged row (padding spreads the banks)
static_assert(BM * STAGE_PITCH * 4 <= OFF_HI_B - OFF_RAW_A, "staged partial tile must fit the raw ring");
static_assert(SPLIT_WARPS * EPI_STAGE_FLOATS * 4 <= OFF_HI_B - OFF_RAW_A, "epilogue staging must fit the raw ring");
constexpr int NUM_BARS = 2 * RAW_STAGES + 2 * COMP_STAGES + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack

struct Params {
  int M, N, K;
  int a_kmajor, b_kmajor;
  int k_tiles, kt_per_split;
  EpiArgs epi;
  int splits;  // K splits = CTAs per cluster (1: no cluster, direct epilogue)
  int* err;
};

// ---- PTX wrappers ----------------------------------------------------------
GPT2_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

GPT2_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

GPT2_DEV void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

GPT2_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One arrival per warp (barriers initialised with a count of warps).  Each
// lane makes its own writes visible first (fence.proxy.async for shared
// memory the tensor core or TMA will read, tcgen05.fence::before_thread_sync
// after TMEM reads); the warp barrier then orders them before lane 0's
// release-arrive.  A per-thread arrive would be 32 serialised atomics on one
// shared-memory word per warp.
GPT2_DEV void mbar_arrive_warp(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

GPT2_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

GPT2_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: returns false (and raises the CTA's abort flag and the
// device error word) if the phase does not complete within g_wait_limit_ns
// of wall time or another role of the CTA has aborted.  try_wait may suspend
// the thread for a hardware-defined interval, so the bound is taken on the
// global timer rather than on a poll count (read every 256th failed poll).
// The limit comes from the constant cache.  A limit below 1 us makes every
// wait give up at its first call, without probing: tests use that to drive
// the timeout path the same way every time.
GPT2_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  const uint64_t limit = g_wait_limit_ns;
  if (limit >= 1000) {
    uint64_t t0 = 0;
    for (uint32_t i = 0;; i++) {
      if (mbar_try_wait(bar, parity)) return true;
      if ((i & 255) == 0) {
        if (*abort_flag) return false;
        uint64_t now = globaltimer_ns();
        if (i == 0) t0 = now;
        else if (now - t0 > limit) break;
      }
    }
  }
  *abort_flag = 1;
  dev_set_error(err, DEV_ERR_TIMEOUT);
  return false;
}

// Drain wait used on the abort path (copies or MMAs already in flight must
// land before the CTA frees its resources); bounded the same way.
GPT2_DEV void mbar_wait_drain(uint64_t* bar, uint32_t parity) {
  uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; i++) {
    if (mbar_try_wait(bar, parity)) return;
    if ((i & 255) == 255 && globaltimer_ns() - t0 > WAIT_LIMIT_NS) return;
  }
}

// Pull a tensor map (a kernel parameter written by the host) into the
// descriptor cache while the CTA sets up, ahead of its first TMA copy.
GPT2_DEV void prefetch_tmap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}

GPT2_DEV void tma_load_2d(void* dst, const CUtensorMap* tm, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(smem_u32(dst)), "l"((uint64_t)tm), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// Cluster helpers: CTA rank, barrier over every thread of the cluster, and
// 16-byte loads from a peer CTA's shared memory (DSMEM).
GPT2_DEV uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

GPT2_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}

GPT2_DEV uint32_t map_peer(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

GPT2_DEV float4 ld_dsmem_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Named barrier 1 over the NT threads of a kernel's epilogue warps (threads
// 64 .. 64+NT-1).  NT must equal the number of threads that reach it: each
// kernel instantiates it with its own epilogue width.
template <int NT>
GPT2_DEV void epi_bar() {
  static_assert(NT % 32 == 0, "whole warps");
  asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory");
}

// Named barrier 1 over NT epilogue threads that also ANDs a predicate across
// them: every thread gets the same answer, so a CTA's epilogue threads take
// one decision together (for instance after a bounded wait that may have
// timed out for some of them).
template <int NT>
GPT2_DEV bool epi_bar_and(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.and.pred po, 1, %2, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NT)
      : "memory");
  return r != 0;
}

GPT2_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
GPT2_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// K-major operand, 128-byte swizzle: 8-row atoms of 1024 bytes (SBO), start
// address in 16-byte units, descriptor version 1, layout type 2 (SWIZZLE_128B).
GPT2_DEV uint64_t smem_desc_kmajor_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)(1024 >> 4) << 32;  // stride byte offset: next 8-row group
  d |= (uint64_t)1 << 46;            // version
  d |= (uint64_t)2 << 61;            // SWIZZLE_128B
  return d;
}

// Instruction descriptor: D fp32, A/B tf32, both K-major, M = 128, N = BN.
constexpr uint32_t IDESC_TF32 = (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(BN >> 3) << 17) |
                                ((uint32_t)(BM >> 4) << 24);

GPT2_DEV void mma_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(IDESC_TF32), "r"(accumulate)
      : "memory");
}

// The same MMA with A read from tensor memory (M rows in TMEM lanes 0..127,
// the instruction's 8 K values in 8 consecutive columns from a_tmem).
GPT2_DEV void mma_tf32_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(IDESC_TF32), "r"(accumulate)
      : "memory");
}

GPT2_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

GPT2_DEV void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int k = 0; k < 32; k++) v[k] = __uint_as_float(r[k]);
}

// ---- 3xTF32 split ----------------------------------------------------------
// hi = x rounded to 10 mantissa bits (nearest, ties away); lo = x - hi exactly.
GPT2_DEV float tf32_hi(float x) { return __uint_as_float((__float_as_uint(x) + 0x1000u) & 0xFFFFE000u); }

GPT2_DEV void split4(float4 x, float4& h, float4& l) {
  h = make_float4(tf32_hi(x.x), tf32_hi(x.y), tf32_hi(x.z), tf32_hi(x.w));
  l = make_float4(x.x - h.x, x.y - h.y, x.z - h.z, x.w - h.w);
}

// 16 consecutive TMEM columns of this warp's 32 lanes from v[] (lane i -> TMEM
// lane (taddr >> 16) + i).  Asynchronous: tcgen05.wait::st before the values
// are handed to the tensor core.
GPT2_DEV void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
      "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
      "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
      : "memory");
}

// A operand into TMEM: this lane holds tile row m (its TMEM lane) and the 16
// K values [16h, 16h + 16); their hi halves go to columns t_hi .. t_hi + 15
// and the lo halves to t_hi + 32 .. (t_hi is this warp's lane base, the
// stage's hi column and 16h).  K-major raw tiles are as TMA wrote them with
// the 128-byte swizzle: the 16-byte chunk c of row m sits at chunk c ^ (m & 7).
GPT2_DEV void split_a_kmajor_tmem(const float* raw, uint32_t t_hi, int m, int h) {
  float hv[16], lv[16];
#pragma unroll
  for (int cc = 0; cc < 4; cc++) {
    const int c = 4 * h + cc;
    float4 hh, ll;
    split4(*reinterpret_cast<const float4*>(raw + m * BK + ((c ^ (m & 7)) << 2)), hh, ll);
    hv[4 * cc] = hh.x; hv[4 * cc + 1] = hh.y; hv[4 * cc + 2] = hh.z; hv[4 * cc + 3] = hh.w;
    lv[4 * cc] = ll.x; lv[4 * cc + 1] = ll.y; lv[4 * cc + 2] = ll.z; lv[4 * cc + 3] = ll.w;
  }
  tmem_st16(t_hi, hv);
  tmem_st16(t_hi + BK, lv);
}

// The same from an MN-major raw tile (unswizzled [BK rows of k][128 of m]).
GPT2_DEV void split_a_mnmajor_tmem(const float* raw, uint32_t t_hi, int m, int h) {
  float hv[16], lv[16];
#pragma unroll
  for (int k = 0; k < 16; k++) {
    const float x = raw[(16 * h + k) * BM + m];
    hv[k] = tf32_hi(x);
    lv[k] = x - hv[k];
  }
  tmem_st16(t_hi, hv);
  tmem_st16(t_hi + BK, lv);
}

// raw tile already K-major SW128 (as TMA wrote it): split in place order.
GPT2_DEV void split_kmajor(const float4* raw, float4* hi, float4* lo, int t) {
#pragma unroll
  for (int j = 0; j < (BM * BK / 4) / SPLIT_THREADS; j++) {
    int q = t + SPLIT_THREADS * j;
    float4 h, l;
    split4(raw[q], h, l);
    hi[q] = h;
    lo[q] = l;
  }
}

// raw tile MN-major, unswizzled [BK rows of k][128 of m]: the two threads
// t and t + 128 own row m = t % 128 and write half of its 32 k-values each
// as swizzled 16-byte chunks.
GPT2_DEV void split_mnmajor(const float* raw, float* hi, float* lo, int t) {
  const int m = t & (BM - 1), c0 = (t / BM) * (BK / 8);
#pragma unroll
  for (int cc = 0; cc < BK / 8; cc++) {
    const int c = c0 + cc;
    float4 x = make_float4(raw[(4 * c + 0) * BM + m], raw[(4 * c + 1) * BM + m], raw[(4 * c + 2) * BM + m],
                           raw[(4 * c + 3) * BM + m]);
    float4 h, l;
    split4(x, h, l);
    int off = m * 32 + ((c ^ (m & 7)) << 2);
    *reinterpret_cast<float4*>(hi + off) = h;
    *reinterpret_cast<float4*>(lo + off) = l;
  }
}

// ---- the kernel -------------------------------------------------------------
__global__ void __launch_bounds__(THREADS, 1)
    gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ Params p) {
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = bars + RAW_STAGES;
  uint64_t* comp_full = bars + 2 * RAW_STAGES;
  uint64_t* comp_empty = bars + 2 * RAW_STAGES + COMP_STAGES;
  uint64_t* acc_full = bars + 2 * RAW_STAGES + 2 * COMP_STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  volatile int* go_flag = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int kt0 = blockIdx.z * p.kt_per_split;
  const int kt1 = min(p.k_tiles, kt0 + p.kt_per_split);
  const int nk = kt1 - kt0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; s++) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], SPLIT_WARPS);
    }
    for (int s = 0; s < COMP_STAGES; s++) {
      mbar_init(&comp_full[s], SPLIT_WARPS);
      mbar_init(&comp_empty[s], 1);
    }
    mbar_init(acc_full, 1);
    *abort_flag = 0;
    *go_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the first global-memory access comes after this

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nk; i++) {
        int s = i % RAW_STAGES;
        uint32_t ph = (i / RAW_STAGES) & 1;
        if (!mbar_wait(&raw_empty[s], ph ^ 1, abort_flag, p.err)) break;
        int k = (kt0 + i) * BK;
        mbar_expect_tx(&raw_full[s], 2 * TILE_BYTES);
        uint8_t* ra = smem + OFF_RAW_A + s * TILE_BYTES;
        uint8_t* rb = smem + OFF_RAW_B + s * TILE_BYTES;
        if (p.a_kmajor) tma_load_2d(ra, &tmA, k, m0, &raw_full[s]);
        else tma_load_2d(ra, &tmA, m0, k, &raw_full[s]);
        if (p.b_kmajor) tma_load_2d(rb, &tmB, k, n0, &raw_full[s]);
        else tma_load_2d(rb, &tmB, n0, k, &raw_full[s]);
        issued = i + 1;
      }
      // on abort, let the copies already in flight land before the CTA exits
      if (*abort_flag) {
        for (int i = max(0, issued - RAW_STAGES); i < issued; i++) {
          int s = i % RAW_STAGES;
          mbar_wait_drain(&raw_full[s], (i / RAW_STAGES) & 1);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      for (int i = 0; i < nk && ok; i++) {
        int c = i % COMP_STAGES;
        uint32_t ph = (i / COMP_STAGES) & 1;
        if (!mbar_wait(&comp_full[c], ph, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ah = tmem + (uint32_t)(TM_A + c * 2 * BK), al = ah + BK;
        const uint32_t bh = smem_u32(smem + OFF_HI_B + c * TILE_BYTES), bl = smem_u32(smem + OFF_LO_B + c * TILE_BYTES);
#pragma unroll
        for (int j = 0; j < BK / 8; j++) {  // kind::tf32 consumes K = 8 (32 bytes, 8 TMEM columns) per instruction
          const uint64_t dbh = smem_desc_kmajor_sw128(bh + j * 32), dbl = smem_desc_kmajor_sw128(bl + j * 32);
          mma_tf32_ta(tmem, ah + 8 * j, dbh, (i > 0 || j > 0) ? 1u : 0u);
          mma_tf32_ta(tmem, ah + 8 * j, dbl, 1u);
          mma_tf32_ta(tmem, al + 8 * j, dbh, 1u);
        }
        mma_commit(&comp_empty[c]);  // frees the hi/lo stage once these MMAs have read it
      }
      // acc_full tracks completion of every MMA this thread issued; on abort
      // wait for it here so that TMEM is not freed under running MMAs
      if (nk > 0) mma_commit(acc_full);
      if (!ok && nk > 0) {
        mbar_wait_drain(acc_full, 0);
      }
    }
  } else {
    // ---------------- splitters, then epilogue ----------------
    const int t = threadIdx.x - 64;  // 0 .. SPLIT_THREADS-1
    // The epilogue's global reads (C for the accumulating product, R for the
    // residual and GELU-derivative products) are only needed after the main
    // loop: start pulling this thread's output row into L2 now.
    if (p.splits == 1 && t < BM && m0 + t < p.M) {
      const float* src = p.epi.epi == EPI_ACCUM ? p.epi.C + (size_t)(m0 + t) * p.epi.ldc
                         : (p.epi.epi == EPI_BIAS_RESID || p.epi.epi == EPI_DGELU) ? p.epi.R + (size_t)(m0 + t) * p.epi.ldr
                                                                                   : nullptr;
      if (src) {
#pragma unroll
        for (int c = 0; c < BN * 4 / 128; c++)
          if (n0 + c * 32 < p.N) asm volatile("prefetch.global.L2 [%0];" ::"l"(src + n0 + c * 32));
      }
    }
    const int a_quad = warp & 3, a_half = (warp - 2) >> 2;  // TMEM lanes this warp may access; its K half
    bool ok = true;
    for (int i = 0; i < nk; i++) {
      int s = i % RAW_STAGES, c = i % COMP_STAGES;
      // one decision per warp: its lanes arrive together below
      if (!__all_sync(0xffffffffu, mbar_wait(&raw_full[s], (i / RAW_STAGES) & 1, abort_flag, p.err) &&
                                       mbar_wait(&comp_empty[c], ((i / COMP_STAGES) & 1) ^ 1, abort_flag, p.err))) {
        ok = false;
        break;
      }
      tc_fence_after();  // the MMAs that read this stage's TMEM columns have completed
      const float* ra = reinterpret_cast<const float*>(smem + OFF_RAW_A + s * TILE_BYTES);
      const uint8_t* rb = smem + OFF_RAW_B + s * TILE_BYTES;
      float* hb = reinterpret_cast<float*>(smem + OFF_HI_B + c * TILE_BYTES);
      float* lb = reinterpret_cast<float*>(smem + OFF_LO_B + c * TILE_BYTES);
      // A: this warp's TMEM lane quadrant, half of the K columns
      const uint32_t t_hi = tmem + ((uint32_t)(a_quad * 32) << 16) + (uint32_t)(TM_A + c * 2 * BK + 16 * a_half);
      if (p.a_kmajor) split_a_kmajor_tmem(ra, t_hi, a_quad * 32 + lane, a_half);
      else split_a_mnmajor_tmem(ra, t_hi, a_quad * 32 + lane, a_half);
      if (p.b_kmajor)
        split_kmajor(reinterpret_cast<const float4*>(rb), reinterpret_cast<float4*>(hb), reinterpret_cast<float4*>(lb), t);
      else
        split_mnmajor(reinterpret_cast<const float*>(rb), hb, lb, t);
      // make the TMEM stores complete and the generic-proxy smem writes
      // visible to the tensor core (async proxy) before the hand-off
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&raw_empty[s]);
        mbar_arrive(&comp_full[c]);
      }
    }
    if (ok && nk > 0) ok = mbar_wait(acc_full, 0, abort_flag, p.err);
    // One decision for all epilogue warps (tcgen05.ld is warp-collective and
    // the split-K hand-off below uses a barrier over these threads).
    // Every epilogue thread reaches this barrier: all of its waits are bounded.
    epi_bar<SPLIT_THREADS>();
    if (t == 0) *go_flag = (nk > 0 && !*abort_flag) ? 1 : 0;
    epi_bar<SPLIT_THREADS>();
    if (*go_flag) {
      tc_fence_after();
      const int q = warp & 3;  // TMEM lane quadrant this warp may access
      const int row = q * 32 + lane;
      const int half = (warp - 2) >> 2;  // which half of the 128 columns this warp finishes
      float* stage = reinterpret_cast<float*>(smem + OFF_STAGE);
#pragma unroll 1
      for (int cc = half * (BN / 64); cc < (half + 1) * (BN / 64); cc++) {
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(cc * 32), v);
        if (p.splits > 1) {
          // this split's partial tile, row-major with a padded pitch, for the cluster reduction
          float* dst = stage + row * STAGE_PITCH + cc * 32;
#pragma unroll
          for (int u = 0; u < 8; u++) st4(dst + 4 * u, make_float4(v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]));
        } else {
          // coalesced epilogue through this warp's staging area (the hi/lo
          // region is free once the accumulator is complete)
          const int j0 = n0 + cc * 32, i0 = m0 + q * 32;
          if (j0 < p.N && i0 < p.M) {  // warp-uniform
            float* ws = reinterpret_cast<float*>(smem + OFF_STAGE) + (warp - 2) * EPI_STAGE_FLOATS;
            warp32_stage(ws, v, lane);
            warp32_epilogue(p.epi, ws, i0, j0, p.M, p.N, lane);
          }
        }
      }
    }
  }

  if (p.splits > 1) {
    // Split-K reduction inside the cluster: the K splits of this output tile
    // are the CTAs of one cluster.  Once every partial is staged, CTA r sums
    // rows [r*R, (r+1)*R) of the tile over the splits in split order, reading
    // the peers' shared memory, and applies the epilogue.  Every thread of
    // every CTA reaches both cluster barriers (all waits above are bounded).
    cluster_sync();
    if (warp >= 2 && *go_flag) {
      const int S = p.splits;
      const int rank = (int)cluster_rank();
      const int R = (BM + S - 1) / S;
      const int r0 = rank * R, r1 = min(BM, r0 + R);
      const int t = threadIdx.x - 64;
      const int c4 = t & 31;  // float4 column group of the 128-wide tile
      const int j = n0 + 4 * c4;
      const uint32_t stage = smem_u32(smem + OFF_STAGE);
      // the bias of this thread's four columns, once; per row, the epilogue's
      // global input is requested before the peers' partials, so its latency
      // overlaps theirs instead of following them
      const bool vec = p.epi.vec4 && j + 4 <= p.N;
      const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
      const float4 bias4 = (vec && epi_has_bias(p.epi.epi)) ? ld4(p.epi.bias + j) : zero;
      for (int r = r0 + (t >> 5); r < r1; r += SPLIT_WARPS) {
        const int ii = m0 + r;
        if (ii >= p.M || j >= p.N) continue;
        const float4 in4 = (vec && epi_has_input(p.epi.epi)) ? epi_load_input(p.epi, ii, j) : zero;
        const uint32_t off = stage + (uint32_t)(r * STAGE_PITCH + 4 * c4) * 4u;
        // every peer's partial is loaded before any is summed (the loads
        // overlap instead of each waiting for the previous one's add)
        float4 part[8];
#pragma unroll
        for (int z = 0; z < 8; z++)
          if (z < S) part[z] = ld_dsmem_f4(map_peer(off, (uint32_t)z));
        float4 acc = part[0];
#pragma unroll
        for (int z = 1; z < 8; z++)
          if (z < S) {
            acc.x += part[z].x; acc.y += part[z].y; acc.z += part[z].z; acc.w += part[z].w;
          }
        if (vec) {
          epi_apply4(p.epi, ii, j, acc, bias4, in4);
        } else if (j + 4 <= p.N) {
          epi_store4(p.epi, ii, j, acc);
        } else {
          const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
          for (int c = 0; c < 4 && j + c < p.N; c++) epi_store(p.epi, ii, j + c, a4[c]);
        }
      }
    }
    cluster_sync();  // peers keep their shared memory until every CTA has read it
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
  }
}

// ---- the persistent variant ---------------------------------------------------
// For products with more 128 x 128 output tiles than SMs and no K split (the
// LM head forward and its weight gradient): one CTA per SM walks the tiles
// (stride gridDim.x), so a tile's TMEM set-up, first copies and epilogue
// overlap the neighbouring tiles' main loops instead of being paid once per
// tile.  The roles are those above plus four epilogue warps; the MMAs
// alternate between two TMEM accumulators (columns 0..127 and 128..255), the
// epilogue warps drain one while the other fills, and A's hi/lo stages sit in
// columns 256..383.  Tiles are numbered with the operand that is reused
// varying fastest: when there are fewer row tiles than column tiles,
// consecutive tiles share a column block of B (read from HBM about once),
// otherwise they share a row block of A.
namespace pers {
constexpr int EPI_WARPS = 4;
constexpr int THREADS = 64 + SPLIT_THREADS + 32 * EPI_WARPS;
constexpr int TMEM_COLS = 512;
constexpr int TM_ACC = 0;    // accumulator b at columns b * BN
constexpr int TM_A = 2 * BN;  // A stage c: hi at TM_A + 64c, lo at TM_A + 64c + 32
static_assert(TM_A + COMP_STAGES * 2 * BK <= TMEM_COLS, "A stages must fit the TMEM allocation");
constexpr int OFF_RAW_A = 0;
constexpr int OFF_RAW_B = OFF_RAW_A + RAW_STAGES * TILE_BYTES;
constexpr int OFF_HI_B = OFF_RAW_B + RAW_STAGES * TILE_BYTES;
constexpr int OFF_LO_B = OFF_HI_B + COMP_STAGES * TILE_BYTES;
constexpr int OFF_EPI = OFF_LO_B + COMP_STAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_EPI + EPI_WARPS * EPI_STAGE_FLOATS * 4;
constexpr int NUM_BARS = 2 * RAW_STAGES + 2 * COMP_STAGES + 4 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory of one CTA");

GPT2_DEV void tile_coords(int tile, int tiles_m, int tiles_n, int& m0, int& n0) {
  int tm, tn;
  if (tiles_m <= tiles_n) {
    tm = tile % tiles_m;
    tn = tile / tiles_m;
  } else {
    tn = tile % tiles_n;
    tm = tile / tiles_n;
  }
  m0 = tm * BM;
  n0 = tn * BN;
}
}  // namespace pers

__global__ void __launch_bounds__(pers::THREADS, 1)
    gemm_tf32x3_persistent_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                  const __grid_constant__ Params p) {
  using namespace pers;
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + pers::OFF_BAR);
  uint64_t* raw_full = bars;
  uint64_t* raw_empty = bars + RAW_STAGES;
  uint64_t* comp_full = bars + 2 * RAW_STAGES;
  uint64_t* comp_empty = bars + 2 * RAW_STAGES + COMP_STAGES;
  uint64_t* acc_full = bars + 2 * RAW_STAGES + 2 * COMP_STAGES;  // [2]
  uint64_t* acc_empty = acc_full + 2;                            // [2]
  uint64_t* mma_done = acc_full + 4;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + pers::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + pers::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles_m = (p.M + BM - 1) / BM, tiles_n = (p.N + BN - 1) / BN;
  const int tiles = tiles_m * tiles_n;
  const int nk = p.k_tiles;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RAW_STAGES; s++) {
      mbar_init(&raw_full[s], 1);
      mbar_init(&raw_empty[s], SPLIT_WARPS);
    }
    for (int s = 0; s < COMP_STAGES; s++) {
      mbar_init(&comp_full[s], SPLIT_WARPS);
      mbar_init(&comp_empty[s], 1);
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(pers::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the first global-memory access comes after this

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
        int m0, n0;
        tile_coords(tile, tiles_m, tiles_n, m0, n0);
        for (int kt = 0; kt < nk; kt++, it++) {
          const int s = it % RAW_STAGES;
          if (!mbar_wait(&raw_empty[s], ((it / RAW_STAGES) & 1) ^ 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          const int k = kt * BK;
          mbar_expect_tx(&raw_full[s], 2 * TILE_BYTES);
          uint8_t* ra = smem + pers::OFF_RAW_A + s * TILE_BYTES;
          uint8_t* rb = smem + pers::OFF_RAW_B + s * TILE_BYTES;
          if (p.a_kmajor) tma_load_2d(ra, &tmA, k, m0, &raw_full[s]);
          else tma_load_2d(ra, &tmA, m0, k, &raw_full[s]);
          if (p.b_kmajor) tma_load_2d(rb, &tmB, k, n0, &raw_full[s]);
          else tma_load_2d(rb, &tmB, n0, k, &raw_full[s]);
        }
      }
      if (!ok) {  // let the copies already in flight land before the CTA exits
        for (int j = max(0, it - RAW_STAGES); j < it; j++) mbar_wait_drain(&raw_full[j % RAW_STAGES], (j / RAW_STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      int it = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x, lt++) {
        const int buf = lt & 1;
        if (!mbar_wait(&acc_empty[buf], ((lt >> 1) & 1) ^ 1, abort_flag, p.err)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(TM_ACC + buf * BN);
        for (int kt = 0; kt < nk; kt++, it++) {
          const int c = it % COMP_STAGES;
          if (!mbar_wait(&comp_full[c], (it / COMP_STAGES) & 1, abort_flag, p.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ah = tmem + (uint32_t)(pers::TM_A + c * 2 * BK), al = ah + BK;
          const uint32_t bh = smem_u32(smem + pers::OFF_HI_B + c * TILE_BYTES);
          const uint32_t bl = smem_u32(smem + pers::OFF_LO_B + c * TILE_BYTES);
#pragma unroll
          for (int j = 0; j < BK / 8; j++) {
            const uint64_t dbh = smem_desc_kmajor_sw128(bh + j * 32), dbl = smem_desc_kmajor_sw128(bl + j * 32);
            mma_tf32_ta(d_tmem, ah + 8 * j, dbh, (kt > 0 || j > 0) ? 1u : 0u);
            mma_tf32_ta(d_tmem, ah + 8 * j, dbl, 1u);
            mma_tf32_ta(d_tmem, al + 8 * j, dbh, 1u);
          }
          mma_commit(&comp_empty[c]);  // frees the hi/lo stage once these MMAs have read it
        }
        if (ok) mma_commit(&acc_full[buf]);
      }
      // every MMA this thread issued has completed once mma_done fires
      mma_commit(mma_done);
      mbar_wait_drain(mma_done, 0);
    }
  } else if (warp < 2 + SPLIT_WARPS) {
    // ---------------- splitters ----------------
    const int t = threadIdx.x - 64;
    const int a_quad = warp & 3, a_half = (warp - 2) >> 2;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      for (int kt = 0; kt < nk; kt++, it++) {
        const int s = it % RAW_STAGES, c = it % COMP_STAGES;
        if (!__all_sync(0xffffffffu, mbar_wait(&raw_full[s], (it / RAW_STAGES) & 1, abort_flag, p.err) &&
                                         mbar_wait(&comp_empty[c], ((it / COMP_STAGES) & 1) ^ 1, abort_flag, p.err))) {
          ok = false;
          break;
        }
        tc_fence_after();  // the MMAs that read this stage's TMEM columns have completed
        const float* ra = reinterpret_cast<const float*>(smem + pers::OFF_RAW_A + s * TILE_BYTES);
        const uint8_t* rb = smem + pers::OFF_RAW_B + s * TILE_BYTES;
        float* hb = reinterpret_cast<float*>(smem + pers::OFF_HI_B + c * TILE_BYTES);
        float* lb = reinterpret_cast<float*>(smem + pers::OFF_LO_B + c * TILE_BYTES);
        const uint32_t t_hi = tmem + ((uint32_t)(a_quad * 32) << 16) + (uint32_t)(pers::TM_A + c * 2 * BK + 16 * a_half);
        if (p.a_kmajor) split_a_kmajor_tmem(ra, t_hi, a_quad * 32 + lane, a_half);
        else split_a_mnmajor_tmem(ra, t_hi, a_quad * 32 + lane, a_half);
        if (p.b_kmajor)
          split_kmajor(reinterpret_cast<const float4*>(rb), reinterpret_cast<float4*>(hb), reinterpret_cast<float4*>(lb), t);
        else
          split_mnmajor(reinterpret_cast<const float*>(rb), hb, lb, t);
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&raw_empty[s]);
          mbar_arrive(&comp_full[c]);
        }
      }
    }
  } else {
    // ---------------- epilogue ----------------
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    float* stage = reinterpret_cast<float*>(smem + pers::OFF_EPI) + (warp - 2 - SPLIT_WARPS) * EPI_STAGE_FLOATS;
    int lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, lt++) {
      int m0, n0;
      tile_coords(tile, tiles_m, tiles_n, m0, n0);
      const int buf = lt & 1;
      // one decision per warp (tcgen05.ld is warp-collective)
      if (!__all_sync(0xffffffffu, mbar_wait(&acc_full[buf], (lt >> 1) & 1, abort_flag, p.err))) break;
      tc_fence_after();
      const int i0 = m0 + q * 32;
      const uint32_t tbase = tmem + (uint32_t)(TM_ACC + buf * BN) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; cc++) {
        float v[32];
        tmem_ld32(tbase + (uint32_t)(cc * 32), v);
        const int j0 = n0 + cc * 32;
        if (j0 < p.N && i0 < p.M) {  // warp-uniform
          warp32_stage(stage, v, lane);
          warp32_epilogue(p.epi, stage, i0, j0, p.M, p.N, lane);
        }
      }
      // the accumulator is in global memory now: hand it back to the MMAs
      tc_fence_before();
      mbar_arrive_warp(&acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(pers::TMEM_COLS) : "memory");
  }
}

}  // namespace tc
