// Fused drafter LM-head + top-K marginals: the logits l_k = W h_k of every
// drafter row are formed on the tensor cores and reduced to step 1's outputs
// (the K best tokens, their logits and lse) without the logits ever reaching
// global memory.
//
// Bastion (gist.science/nl/paper/2605.29727), Methodologie §1: one forward
// pass of the block-diffusion drafter yields the position-wise marginals
// q_k = softmax(l_k); its last layer is the output embedding W applied to the
// final hidden state h_k of each block position.
//
// sm_103a design (one persistent CTA per SM):
//  * the rows are cut into M-tiles of 128 and the vocabulary into N-tiles of
//    192; CTA c owns M-tile c % MT and every CPM-th N-tile from c / MT on, so
//    the MT CTAs that read the same N-tile of W run side by side and W comes
//    from HBM about once (the other reads hit L2; optionally the MT CTAs form
//    a cluster and each loads a slice of the W tile for all of them);
//  * warp 0 streams A (hidden, 128 x 64) and B (W, 192 x 64) tiles through a
//    4-stage ring with TMA (cp.async.bulk.tensor, 128-byte swizzle, zero fill
//    past the edges); lane 0 of warp 1 issues tcgen05.mma kind::f16 (bf16 in,
//    fp32 accumulate, M = 128, N = 192, K = 16, four per 64-column chunk)
//    into one of two TMEM accumulators of 192 columns, so the epilogue of one
//    tile overlaps the MMAs of the next.  (N = 192 rather than 256 leaves
//    shared memory for a fourth stage next to the heaps; three stages of
//    N = 256 left the MMAs waiting for operands);
//  * warps 2-5 are the epilogue, one thread per row (TMEM lane): per 32-column
//    chunk (tcgen05.ld) the thread updates its row's running max and sum of
//    2^(l log2(e) - c) (c an integer kept at floor(max log2(e)), the sum
//    rescaled by exact powers of two) and inserts every logit whose key
//    (value desc, token asc, one 64-bit integer) beats the root of the row's
//    4-ary min-heap of the K best keys seen (in shared memory, one column of
//    heap slots per thread; the first K keys are stored as they come and the
//    heap is built once) and above the row's bound.  Each share keeps its 4
//    best keys exactly and publishes the 4th; the bound is the m-th largest
//    published value, m = ceil(K / 4): m shares hold 4 keys each at or above
//    it, so a key below it cannot be among the row's K best and is not
//    inserted.  The first tile is read twice from TMEM: first for the 4 best,
//    the max and the sum, then, once m shares have published (a bounded wait
//    of at most ~20 us, while the MMAs fill the other accumulator), for the
//    heap; the bound is read again after the next tiles.  (Filling the heap
//    before a bound existed inserted about half of the first tile's columns
//    and most of the epilogue's time went to heap sifts.)  The heap then holds
//    every key of the share that can be among the row's K best;
//  * a merge kernel takes, per row, the CPM heaps (radix selection of the K-th
//    best key over them, then ranking by counting) and the CPM (max, c, sum)
//    shares (exact powers of two again), and writes the K best logits, tokens,
//    log q and lse.
// Every wait is bounded (~1 s); on a timeout the CTA flags the rows' requests,
// lets its copies and MMAs end (bounded), frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdlib>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kLT = 192;  // warp 0 TMA, warp 1 MMA (and TMEM), warps 2-5 epilogue
constexpr int kBM = 128, kBN = 192, kBK = 64;
constexpr int kStages = 4;
constexpr int kMaxK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;             // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;             // 24 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;     // 40 KB (a multiple of 1 KB)
constexpr uint32_t kOffHeap = kStages * kStageBytes;    // heaps after the ring
constexpr uint32_t kHeapBytes = kBM * kMaxK * 8;        // 64 KB
constexpr uint32_t kOffBar = kOffHeap + kHeapBytes;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;        // + alignment slack
constexpr float kL2e = 1.4426950216293335f;             // log2(e) rounded to float
constexpr float kCNone = -1.0e30f;                      // c before the first finite logit

struct LmArgs {
  int rows, H, V, K, b, MT, NT, CPM, KC, J;
  int CL;  // CTAs of a cluster: M-tiles that share each W tile, loaded once and multicast
  uint64_t *part_keys;  // [rows][CPM][K]
  float4 *part_stat;    // [rows][CPM]: max, c, sum (hi, lo)
  uint64_t *pub;        // [rows][CPS]: each share's J-th (4th) best key so far (0: none yet);
                        // CPS = CPM rounded up to even, so each row's slots are 16-byte aligned
  int32_t *status;
};

struct LmBars {
  uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], mma_done;
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)(16u >> 4) << 16;    // leading byte offset (unused with the swizzle)
  d |= (uint64_t)(1024u >> 4) << 32;  // stride byte offset: 8 rows of 128 bytes
  d |= (uint64_t)1 << 46;             // descriptor version
  d |= (uint64_t)2 << 61;             // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B (both
// K-major), M = 128, N = 192.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kBN >> 3) << 17) |
                            ((uint32_t)(kBM >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(kIdesc), "r"(accum));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Arrives on the same barrier of every CTA in mask once this thread's MMAs
// so far have completed.
__device__ __forceinline__ void mma_commit_mc(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(mask)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// tcgen05.ld of 32 columns without waiting, and a wait tied to the
// destination registers (so no use of them is scheduled before it).
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_tied(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                 "+r"(r[31])
               :
               : "memory");
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Sum of 2^(x_i k + nc) over four values: two packed f32x2 FMAs, four ex2,
// one packed add; the pair (s0, s1) accumulates.
__device__ __forceinline__ void exp4_acc(float x0, float x1, float x2, float x3, float k, float nc,
                                         float &s0, float &s1) {
  float t0, t1, t2, t3;
  asm("{\n .reg .b64 d, e, kk, cc;\n"
      " mov.b64 d, {%4, %5};\n mov.b64 e, {%6, %7};\n mov.b64 kk, {%9, %9};\n"
      " mov.b64 cc, {%8, %8};\n fma.rn.f32x2 d, d, kk, cc;\n fma.rn.f32x2 e, e, kk, cc;\n"
      " mov.b64 {%0, %1}, d;\n mov.b64 {%2, %3}, e;\n}\n"
      : "=f"(t0), "=f"(t1), "=f"(t2), "=f"(t3)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3), "f"(nc), "f"(k));
  float e0, e1, e2, e3;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(t0));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(t1));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e2) : "f"(t2));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e3) : "f"(t3));
  asm("{\n .reg .b64 a, b, c;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " mov.b64 c, {%4, %5};\n add.rn.f32x2 a, a, b;\n add.rn.f32x2 a, a, c;\n"
      " mov.b64 {%0, %1}, a;\n}\n"
      : "+f"(s0), "+f"(s1)
      : "f"(e0), "f"(e1), "f"(e2), "f"(e3));
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

// The same box into the same shared-memory offset of every CTA in mask, each
// CTA's barrier at bar's offset counting the bytes.
__device__ __forceinline__ void tma_load_2d_mc(void *dst, const CUtensorMap *map, int c0, int c1,
                                               uint64_t *bar, uint16_t mask) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2^d for an integer-valued d <= 0 (0 below the normal range).
__device__ __forceinline__ float pow2_int(float d) {
  return d < -126.f ? 0.f : __int_as_float(((int)d + 127) << 23);
}

__device__ __forceinline__ float2 two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return make_float2(s, (a - (s - bb)) + (b - bb));
}

// Bounded wait that also honours the CTA's abort flag; a wait that runs out
// sets the flag and the request's timeout bit.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         int32_t *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  uint32_t spins = 0;
  while (!mbar_try_wait(bar, parity)) {
    if ((++spins & 63u) == 0u) {
      if (*abort) return false;
      if (global_ns() - t0 > 1000000000ull) {
        *abort = 1;
        atomicOr(status, BASTION_STATUS_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Thread rl's min-heap of K keys: slot i at byte i * kBM * 8 + rl * 8 from
// heap_base (a shared-memory address), so a warp's threads touch consecutive
// words of a slot row.
__device__ __forceinline__ uint64_t hp_ld(uint32_t a) {
  uint64_t v;
  asm volatile("ld.shared.u64 %0, [%1];" : "=l"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void hp_st(uint32_t a, uint64_t v) {
  asm volatile("st.shared.u64 [%0], %1;" ::"r"(a), "l"(v) : "memory");
}

// Sifts key down from slot pos of the heap (slot pos is being replaced).  The
// heap is 4-ary (children of slot p: 4p + 1 .. 4p + 4): three levels for 64
// keys, the four children of a level loaded together.
__device__ __forceinline__ void heap_sift(uint32_t hb, int K, int pos, uint64_t key) {
  constexpr uint32_t kRow = kBM * 8;
  while (true) {
    const int c0 = 4 * pos + 1;
    if (c0 >= K) break;
    uint64_t h[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) h[u] = c0 + u < K ? hp_ld(hb + (uint32_t)(c0 + u) * kRow) : ~0ull;
    int ch = c0;
    uint64_t hc = h[0];
#pragma unroll
    for (int u = 1; u < 4; ++u)
      if (h[u] < hc) {
        hc = h[u];
        ch = c0 + u;
      }
    if (hc >= key) break;
    hp_st(hb + (uint32_t)pos * kRow, hc);
    pos = ch;
  }
  hp_st(hb + (uint32_t)pos * kRow, key);
}

// Builds thread rl's heap from its K stored slots (once per share).
__device__ __noinline__ void heap_build(uint32_t hb, int K) {
  for (int i = (K - 2) / 4; i >= 0; --i) heap_sift(hb, K, i, hp_ld(hb + (uint32_t)i * (kBM * 8)));
}

__global__ void __launch_bounds__(kLT, 1)
    lm_head_kernel(const __grid_constant__ CUtensorMap tm_h, const __grid_constant__ CUtensorMap tm_w,
                   LmArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  LmBars &bs = *reinterpret_cast<LmBars *>(smem + kOffBar);
  uint64_t *heap = reinterpret_cast<uint64_t *>(smem + kOffHeap);  // [K][128]
  volatile int *abort = &bs.abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x % a.MT, j0 = blockIdx.x / a.MT;
  const int ntile = j0 < a.NT ? (a.NT - j0 + a.CPM - 1) / a.CPM : 0;  // N-tiles of this CTA
  const int steps = ntile * a.KC;
  // the request of the CTA's first row takes a timeout bit (rows past the
  // batch never get one)
  int32_t *st0 = &a.status[min(mt * kBM, a.rows - 1) / a.b];

  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_h)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_w)) : "memory");
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bs.full[s], 1);
      mbar_init(&bs.empty[s], (uint32_t)a.CL);  // every CTA of the cluster has read the stage
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bs.acc_full[s], 1);
      mbar_init(&bs.acc_empty[s], 4);  // one arrival per epilogue warp
    }
    mbar_init(&bs.mma_done, 1);
    bs.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&bs.tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the heaps start as K zero keys: zero is below every real key
  for (int i = tid; i < kBM * a.K; i += kLT) heap[i] = 0ull;
  griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs.tmem;
  // every CTA of the cluster has set its barriers before any copy or commit
  // reaches them
  const uint16_t cmask = (uint16_t)((1u << a.CL) - 1u);
  const int crank = blockIdx.x % a.CL;
  if (a.CL > 1) {
    cluster_arrive_relaxed();
    cluster_wait();
  }

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int g = 0; g < steps; ++g) {
        const int s = g % kStages;
        if (g >= kStages && !wait_bar(&bs.empty[s], (uint32_t)((g / kStages) - 1) & 1u, abort, st0)) break;
        const int t = g / a.KC, kc = g - t * a.KC;
        const int n = j0 + t * a.CPM;
        unsigned char *dst = smem + (uint32_t)s * kStageBytes;
        mbar_arrive_expect_tx(&bs.full[s], kStageBytes);
        tma_load_2d(dst, &tm_h, kc * kBK, mt * kBM, &bs.full[s]);
        if (a.CL == 1) {
          tma_load_2d(dst + kABytes, &tm_w, kc * kBK, n * kBN, &bs.full[s]);
        } else {  // this CTA's slice of the W tile, into every CTA of the cluster
          const int sr = kBN / a.CL;
          tma_load_2d_mc(dst + kABytes + (uint32_t)(crank * sr) * 128u, &tm_w, kc * kBK, n * kBN + crank * sr,
                         &bs.full[s], cmask);
        }
        issued = g + 1;
      }
      // our copies have landed (bounded) before the CTA may exit
      for (int g = issued > kStages ? issued - kStages : 0; g < issued; ++g)
        mbar_wait_bounded(&bs.full[g % kStages], (uint32_t)(g / kStages) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = true;
      for (int t = 0; ok && t < ntile; ++t) {
        const int buf = t & 1;
        if (t >= 2 && !wait_bar(&bs.acc_empty[buf], (uint32_t)((t >> 1) - 1) & 1u, abort, st0)) break;
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)buf * kBN;
        for (int kc = 0; kc < a.KC; ++kc) {
          const int g = t * a.KC + kc, s = g % kStages;
          if (!wait_bar(&bs.full[s], (uint32_t)(g / kStages) & 1u, abort, st0)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (uint32_t)s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int ks = 0; ks < kBK / 16; ++ks)
            mma_bf16(d, sw128_desc(sa + (uint32_t)ks * 32u), sw128_desc(sb + (uint32_t)ks * 32u),
                     (kc > 0 || ks > 0) ? 1u : 0u);
          // the stage frees (in every CTA of the cluster) once these MMAs have read it
          if (a.CL == 1) mma_commit(&bs.empty[s]);
          else mma_commit_mc(&bs.empty[s], cmask);
        }
        if (ok) mma_commit(&bs.acc_full[buf]);
      }
      // every MMA issued has completed (bounded) before the TMEM is freed
      mma_commit(&bs.mma_done);
      mbar_wait_bounded(&bs.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32 quad .. 32 quad + 31
    const int rl = quad * 32 + lane;  // row of the tile = TMEM lane
    const int row = mt * kBM + rl;
    const bool live = row < a.rows;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    float m = -INFINITY, c = kCNone, hi = 0.f, lo = 0.f;
    uint64_t root = 0ull;
    bool bad = false;
    const int K = a.K;
    const uint32_t hb = smem_u32(heap) + (uint32_t)rl * 8u;  // this thread's heap column
    int filled = 0;  // keys stored before the heap is built (the first K)
    // the J best keys of this share so far (J <= 4; 0 where fewer were seen),
    // and lb: a lower bound on the row's K-th best key, as last read
    uint64_t top[4] = {0ull, 0ull, 0ull, 0ull};
    uint64_t lb = 0ull;
    const int J = a.J;
    uint64_t *pub_row = a.pub + (size_t)(live ? row : 0) * (size_t)((a.CPM + 1) & ~1);
    // The row's bound from the shares' published J-th best keys: if m =
    // ceil(K / J) shares have a J-th best >= x, at least K keys of the row are
    // >= x, so no key below x is among the row's K best.  x = the m-th largest
    // published value (m <= 16 with J = 4 and K <= 64); a share that has not
    // published yet reads as 0, so the bound exists once m shares have
    // published.  The row's slots are read as 16-byte words, all loads issued
    // first.
    const int mJ = J > 0 ? (K + J - 1) / J : 1;
    // The selection runs on the keys' value words (32-bit min / max): the
    // bound is the m-th largest value with the lowest tie bits, at most the
    // m-th largest key, so still valid.
    auto read_bound = [&]() -> uint64_t {
      uint32_t big[16];  // the largest published values, descending
#pragma unroll
      for (int i = 0; i < 16; ++i) big[i] = 0u;
      const ulonglong2 *pr = reinterpret_cast<const ulonglong2 *>(pub_row);
#pragma unroll 1
      for (int q0 = 0; q0 < a.CPM; q0 += 32) {
        ulonglong2 w[16];
#pragma unroll
        for (int u = 0; u < 16; ++u)
          w[u] = q0 + 2 * u < a.CPM ? __ldcg(pr + q0 / 2 + u) : make_ulonglong2(0ull, 0ull);
#pragma unroll
        for (int u = 0; u < 32; ++u) {
          const uint32_t x = (u & 1) ? (q0 + u < a.CPM ? (uint32_t)(w[u >> 1].y >> 32) : 0u)
                                     : (uint32_t)(w[u >> 1].x >> 32);
#pragma unroll
          for (int i = 15; i > 0; --i) big[i] = max(big[i], min(big[i - 1], x));
          big[0] = max(big[0], x);
        }
      }
      uint32_t r = big[0];
#pragma unroll
      for (int i = 1; i < 16; ++i) r = i == mJ - 1 ? big[i] : r;
      return (uint64_t)r << 32;
    };
    auto publish = [&]() {
      const uint64_t tj = J == 1 ? top[0] : J == 2 ? top[1] : J == 3 ? top[2] : top[3];
      __stcg(reinterpret_cast<unsigned long long *>(pub_row + j0), (unsigned long long)tj);
    };
    for (int t = 0; t < ntile; ++t) {
      const int buf = t & 1;
      if (!__all_sync(kFull, wait_bar(&bs.acc_full[buf], (uint32_t)(t >> 1) & 1u, abort, st0))) break;
      tc_fence_after();
      const int n = j0 + t * a.CPM;
      const uint32_t tbase = lane_base + (uint32_t)buf * kBN;
      // The first tile runs twice over its accumulator: first the share's J
      // best and the row's max and sum only, then (once the other shares have
      // published theirs: the bound) the heap.  Filling the heap before any
      // bound existed inserted most of the first tile's columns.
      const bool split = t == 0 && J > 0;
      for (int ph = 0; ph < (split ? 2 : 1); ++ph) {
        const bool sums = ph == 0, track = !split || ph == 0, heap_on = !split || ph == 1;
        // chunk cc + 1 is loaded from TMEM while chunk cc is processed
        uint32_t ra[32], rb[32];
        tmem_ld32_issue(tbase, ra);
        tmem_wait_tied(ra);
        for (int cc = 0; cc < kBN / 32; ++cc) {
          if (cc + 1 < kBN / 32) tmem_ld32_issue(tbase + (uint32_t)(cc + 1) * 32u, rb);
          float v[32];
#pragma unroll
          for (int q = 0; q < 32; ++q) v[q] = __uint_as_float(ra[q]);
          const int col0 = n * kBN + cc * 32;
          const int nv = min(32, a.V - col0);  // columns past the vocabulary are zero fill
          if (live && nv > 0) {
            // the chunk's max (NaN ignored: a NaN or +inf logit shows in the
            // sum or the max, checked once at the end)
            float cm;
            if (nv == 32) {
              float m3[11];
#pragma unroll
              for (int q = 0; q < 10; ++q) m3[q] = max3(v[3 * q], v[3 * q + 1], v[3 * q + 2]);
              m3[10] = fmaxf(v[30], v[31]);
              cm = max3(max3(m3[0], m3[1], m3[2]), max3(m3[3], m3[4], m3[5]), max3(m3[6], m3[7], m3[8]));
              cm = max3(cm, m3[9], m3[10]);
            } else {
              cm = -INFINITY;
#pragma unroll
              for (int q = 0; q < 32; ++q)
                if (q < nv) cm = fmaxf(cm, v[q]);
            }
            if (sums) {
              m = fmaxf(m, cm);
              if (m > -INFINITY && m < INFINITY) {
                const float cn = floorf(m * kL2e);
                if (cn > c) {  // exact rescale of the running sum by 2^(c - cn)
                  const float f = c > kCNone ? pow2_int(c - cn) : 0.f;
                  hi *= f;
                  lo *= f;
                  c = cn;
                }
                float s0 = 0.f, s1 = 0.f;
                if (nv == 32) {
#pragma unroll
                  for (int q = 0; q < 32; q += 4) exp4_acc(v[q], v[q + 1], v[q + 2], v[q + 3], kL2e, -c, s0, s1);
                } else {
#pragma unroll
                  for (int q = 0; q < 32; ++q)
                    if (q < nv) s0 += ex2(fmaf(v[q], kL2e, -c));
                }
                const float2 ts = two_sum(hi, s0 + s1);
                hi = ts.x;
                lo += ts.y;
              }
            }
            // The columns that can matter: for the heap, a key above both
            // the heap's root (the K-th best of the share so far; nothing
            // while the heap fills) and the row's bound; for the share's J
            // best (not in the first tile's second pass), a key above its J-th
            // best.  One pass over the chunk's passing columns does both.
            // The chunk is copied to the thread's local memory only when a
            // column passes, and the passing columns are handled in one small
            // loop (a loop unrolled over the 32 columns with the heap code
            // inlined in each copy ran several times slower).
            // The share's J best are kept exactly (every key above its J-th
            // best), so the published values keep rising with the bound.
            const uint64_t tj = J == 1 ? top[0] : J == 2 ? top[1] : J == 3 ? top[2] : top[3];
            const float thr_h = heap_on ? fmaxf(filled < K || root == 0ull ? -INFINITY : key_value(root),
                                                lb == 0ull ? -INFINITY : key_value(lb))
                                        : INFINITY;
            const float thr_t = track && J > 0 ? (tj == 0ull ? -INFINITY : key_value(tj)) : INFINITY;
            const float thr = fminf(thr_h, thr_t);
            uint32_t pass = 0u;
            float stg[32];  // the chunk, copied (to the thread's local memory) only when a column passes
            if (cm >= thr) {
#pragma unroll
              for (int q = 0; q < 32; ++q) pass |= (q < nv && v[q] >= thr ? 1u : 0u) << q;
              if (pass) {
#pragma unroll
                for (int q = 0; q < 32; ++q) stg[q] = v[q];
              }
            }
#pragma unroll 1
            while (pass) {
              const int q = __ffs(pass) - 1;
              pass &= pass - 1u;
              const uint64_t key = make_key(stg[q], (uint32_t)(col0 + q));
              if (track && J > 0) {  // the share's J best
                uint64_t x = key;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  if (i < J && x > top[i]) {
                    const uint64_t y = top[i];
                    top[i] = x;
                    x = y;
                  }
              }
              if (!heap_on || key < lb) continue;  // lb itself is a key of the row: kept
              if (filled < K) {
                hp_st(hb + (uint32_t)filled * (kBM * 8), key);
                if (++filled == K) {
                  heap_build(hb, K);
                  root = hp_ld(hb);
                }
              } else if (key > root) {
                heap_sift(hb, K, 0, key);
                root = hp_ld(hb);
              }
            }
          }
          if (cc + 1 < kBN / 32) {
            tmem_wait_tied(rb);
#pragma unroll
            for (int q = 0; q < 32; ++q) ra[q] = rb[q];
          }
        }
        if (split && ph == 0 && live) {
          // publish the first tile's J best, then read the bound; the other
          // shares finish their first tile at about the same time, so wait
          // (at most ~20 us, while the MMAs fill the other accumulator) until
          // m of them have published
          publish();
          const uint64_t t_end = global_ns() + 20000ull;
          for (;;) {
            const uint64_t x = read_bound();
            if (x != 0ull || global_ns() > t_end) {
              lb = x > lb ? x : lb;
              break;
            }
            __nanosleep(256);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs.acc_empty[buf]);
      // later tiles: publish and read the bound after tiles 1, 3, 7 and 15
      // (each read is a round trip to L2 in the epilogue's path; after
      // every tile: 608 against ~560 us)
      if (live && J > 0 && t > 0 && (t & (t + 1)) == 0) {
        publish();
        const uint64_t x = read_bound();
        lb = x > lb ? x : lb;
      }
    }
    bad = m == INFINITY || !(hi == hi) || !(lo == lo) || hi == INFINITY;
    if (live) {  // this CTA's share of the row: its K best keys and (max, c, sum)
      if (bad) atomicOr(&a.status[row / a.b], BASTION_STATUS_NONFINITE);
      const size_t slot = (size_t)row * a.CPM + j0;
      uint64_t *dst = a.part_keys + slot * K;
      // slots never filled (a share of fewer than K columns) keep their zero keys
      for (int i = 0; i < K; ++i) dst[i] = hp_ld(hb + (uint32_t)i * (kBM * 8));
      a.part_stat[slot] = make_float4(m, c, hi, lo);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
  // no copy or commit of another CTA of the cluster targets this one any more
  if (a.CL > 1) {
    cluster_arrive();
    cluster_wait();
  }
}

// ---------------------------------------------------------------------------- merge
constexpr int kMT = 256;  // threads of the merge kernel

struct MergeArgs {
  const uint64_t *part_keys;
  const float4 *part_stat;
  uint64_t *pub;
  int rows, K, CPM, b;
  float *topk_logq, *topk_logit;
  int32_t *topk_tok;
  double *lse;
  int32_t *status;
};

// Per row: the K best of the CPM shares' keys (radix selection of the K-th
// best key, 8 bits a pass over the 64-bit keys, then every key at or above it)
// and lse from the shares' (max, c, sum).
__global__ void __launch_bounds__(kMT) lm_head_merge_kernel(MergeArgs a) {
  extern __shared__ __align__(16) unsigned char msmem[];
  uint64_t *keys = reinterpret_cast<uint64_t *>(msmem);  // [CPM * K]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t info[2];
  __shared__ uint32_t n_sel;
  __shared__ uint64_t sel[kMaxK];
  __shared__ double s_lse;
  const int tid = threadIdx.x, lane = tid & 31;
  const int row = blockIdx.x;
  const int n = a.CPM * a.K;
  griddep_wait();
  griddep_launch_dependents();
  const uint64_t *src = a.part_keys + (size_t)row * n;
  for (int i = tid; i < n; i += kMT) keys[i] = src[i];
  if (a.pub) {  // the shares' bounds start at zero in the next call
    const int cps = (a.CPM + 1) & ~1;
    for (int i = tid; i < cps; i += kMT) a.pub[(size_t)row * cps + i] = 0ull;
  }
  if (tid == 0) n_sel = 0u;
  // lse: the shares in units of 2^(l log2(e) - c_max), exact powers of two
  if (tid < 32) {
    float M = -INFINITY, cM = kCNone;
    for (int q = lane; q < a.CPM; q += 32) {
      const float4 p = a.part_stat[(size_t)row * a.CPM + q];
      M = fmaxf(M, p.x);
      cM = fmaxf(cM, p.y);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
      cM = fmaxf(cM, __shfl_xor_sync(kFull, cM, o));
    }
    double s = 0.0;
    for (int q = lane; q < a.CPM; q += 32) {
      const float4 p = a.part_stat[(size_t)row * a.CPM + q];
      if (p.y > kCNone) s += ((double)p.z + (double)p.w) * (double)pow2_int(p.y - cM);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if (lane == 0) {
      // sum_i 2^(l_i kL2e - cM), with log2(e) = kL2e + (log2(e) - kL2e): the
      // terms that matter have l_i within a few units of M
      constexpr double kLn2 = 0.6931471805599453;
      const double l2e_lo = 1.4426950408889634 - (double)kL2e;
      double lse = (double)cM * kLn2 + log(s) + (double)M * l2e_lo * kLn2;
      int stt = 0;
      if (!(M > -INFINITY)) stt |= BASTION_STATUS_EMPTY_ROW;
      if (M == INFINITY || !(s == s) || !(s < INFINITY)) stt |= BASTION_STATUS_NONFINITE;
      if (stt) atomicOr(&a.status[row / a.b], stt);
      a.lse[row] = lse;
      s_lse = lse;
    }
  }
  __syncthreads();
  // radix selection of the K-th largest key, 8 bits a pass from the top
  uint64_t prefix = 0ull, pmask = 0ull;
  uint32_t need = (uint32_t)a.K;
  for (int shift = 56; shift >= 0; shift -= 8) {
    hist[tid] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kMT) {
      const uint64_t k = keys[i];
      if ((k & pmask) == prefix) atomicAdd(&hist[(uint32_t)(k >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (tid < 32) {  // scanning the 256 bins from the top
      uint32_t cnt[8], tot = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) { cnt[q] = hist[255 - 8 * lane - q]; tot += cnt[q]; }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t above = incl - tot;
      if (above < need && incl >= need) {
        uint32_t run = above;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (run + cnt[q] >= need) {
            info[0] = 255u - 8u * lane - q;
            info[1] = run;
            break;
          }
          run += cnt[q];
        }
      }
    }
    __syncthreads();
    prefix |= (uint64_t)info[0] << shift;
    pmask |= 255ull << shift;
    need -= info[1];
    __syncthreads();
  }
  // prefix is the K-th largest key (keys are unique): the K keys >= it
  for (int i = tid; i < n; i += kMT) {
    const uint64_t k = keys[i];
    if (k >= prefix) {
      const uint32_t at = atomicAdd(&n_sel, 1u);
      if (at < (uint32_t)a.K) sel[at] = k;
    }
  }
  __syncthreads();
  const int K = a.K;
  if (tid < K) {
    const uint64_t k = sel[tid];
    int r = 0;
    for (int q = 0; q < K; ++q) r += sel[q] > k;
    const size_t o = (size_t)row * K + r;
    const float v = key_value(k);
    a.topk_logit[o] = v;
    a.topk_tok[o] = (int32_t)key_token(k);
    if (a.topk_logq) a.topk_logq[o] = (float)((double)v - s_lse);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

// A 2-D bf16 tensor map over a row-major [d1][d0] matrix, boxes of b1 rows
// of 64 elements (128 bytes, the swizzle width), zero fill past the edges.
bool make_map_2d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint32_t b1) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {d0, d1};
  cuuint64_t strides[1] = {d0 * 2};
  cuuint32_t box[2] = {64, b1};
  cuuint32_t es[2] = {1, 1};
  CUresult rc = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

struct LmPlan {
  int MT, NT, CPM, CL, grid;
};

// Clusters of CL CTAs (M-tiles that share each W tile, loaded once and
// multicast; BASTION_LMHEAD_CLUSTER=2|4 chooses them, the default is none:
// on the batched workload clusters of 2 and 4 measured 669 and 710 us against
// 647 us without, the cluster placement leaving SMs idle), as many as can be
// resident at once.
LmPlan lm_plan(int rows, int V) {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  LmPlan p;
  p.MT = (rows + kBM - 1) / kBM;
  p.NT = (V + kBN - 1) / kBN;
  const char *env = getenv("BASTION_LMHEAD_CLUSTER");
  int want = env ? atoi(env) : 1;
  p.CL = 1;
  for (int cl = 4; cl >= 2; cl /= 2)
    if (cl <= want && p.MT % cl == 0) {
      p.CL = cl;
      break;
    }
  int slots = sms;  // CTAs resident at once (one per SM)
  if (p.CL > 1) {
    cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.CL * sms));
    cfg.blockDim = dim3(kLT);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.CL;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nc = 0;
    if (cudaOccupancyMaxActiveClusters(&nc, lm_head_kernel, &cfg) == cudaSuccess && nc > 0) {
      slots = nc * p.CL;
    } else {
      cudaGetLastError();
      p.CL = 1;
    }
  }
  p.CPM = slots / p.MT;
  if (p.CPM < 1) p.CPM = 1;
  if (p.CPM > p.NT) p.CPM = p.NT;
  p.grid = p.MT * p.CPM;
  return p;
}

}  // namespace

size_t lm_head_workspace_bytes(int rows, int V, int K) {
  const LmPlan p = lm_plan(rows, V);
  const size_t keys = (size_t)rows * p.CPM * K * 8;
  const size_t stat = (size_t)rows * p.CPM * 16;
  const size_t pub = (size_t)rows * ((p.CPM + 1) & ~1) * 8;
  return (keys + 255) / 256 * 256 + (stat + 255) / 256 * 256 + (pub + 255) / 256 * 256;
}

int launch_lm_head(const void *hidden, const void *weight, int B, int b, int H, int V, int K,
                   float *topk_logq, float *topk_logit, int32_t *topk_tok, double *lse, void *ws,
                   int32_t *status, cudaStream_t stream) {
  const int rows = B * b;
  const LmPlan p = lm_plan(rows, V);
  CUtensorMap mh, mw;
  if (!make_map_2d(&mh, hidden, (uint64_t)H, (uint64_t)rows, kBM) ||
      !make_map_2d(&mw, weight, (uint64_t)H, (uint64_t)V, (uint32_t)(kBN / p.CL)))
    return BASTION_ERR_LAUNCH;
  LmArgs a;
  a.rows = rows;
  a.H = H;
  a.V = V;
  a.K = K;
  a.b = b;
  a.MT = p.MT;
  a.NT = p.NT;
  a.CPM = p.CPM;
  a.CL = p.CL;
  a.KC = H / kBK;
  unsigned char *w = static_cast<unsigned char *>(ws);
  const size_t keys = ((size_t)rows * p.CPM * K * 8 + 255) / 256 * 256;
  const size_t stat = ((size_t)rows * p.CPM * 16 + 255) / 256 * 256;
  a.part_keys = reinterpret_cast<uint64_t *>(w);
  a.part_stat = reinterpret_cast<float4 *>(w + keys);
  a.pub = reinterpret_cast<uint64_t *>(w + keys + stat);
  // each share publishes its J = 4th best key: the row's bound needs m =
  // ceil(K / 4) <= 16 shares (K <= 64); none where K > 4 CPM (m > CPM)
  a.J = (K + 3) / 4 <= p.CPM ? 4 : 0;
  a.status = status;
  cudaError_t e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e == cudaSuccess) {
    if (p.CL > 1)
      e = launch_cluster_pdl(lm_head_kernel, dim3((unsigned)p.grid), dim3(kLT), kSmem, stream, p.CL, mh, mw, a);
    else
      e = launch_pdl(lm_head_kernel, dim3((unsigned)p.grid), dim3(kLT), kSmem, stream, mh, mw, a);
  }
  if (e != cudaSuccess) return BASTION_ERR_LAUNCH;
  MergeArgs m;
  m.part_keys = a.part_keys;
  m.part_stat = a.part_stat;
  m.pub = a.pub;
  m.rows = rows;
  m.K = K;
  m.CPM = p.CPM;
  m.b = b;
  m.topk_logq = topk_logq;
  m.topk_logit = topk_logit;
  m.topk_tok = topk_tok;
  m.lse = lse;
  m.status = status;
  const size_t msm = (size_t)p.CPM * K * 8;
  e = cudaFuncSetAttribute(lm_head_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msm);
  if (e == cudaSuccess) e = launch_pdl(lm_head_merge_kernel, dim3((unsigned)rows), dim3(kMT), msm, stream, m);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
