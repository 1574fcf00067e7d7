// Tree-masked GQA attention of the draft tree's query tokens against the KV
// cache: the target's one parallel verification pass over the whole tree
// (Bastion, gist.science/nl/paper/2605.29727, "Probleemstelling": the target
// verifies the drafted candidates in parallel; Methodologie §2: the tree is
// verified as one prefix tree).  Query i sees every committed context slot and
// the tree slots of its own root path (ancestor-or-self bitmask).
//
// sm_103a design, one CTA per (request, KV head, 128 query rows):
//  * the 128 rows are (tree node, query head of the KV group) pairs, so the G
//    heads that share a KV head share every K/V tile read;
//  * thread 0 issues Q and the first two K and V tiles right after the
//    barrier initialisation, before the tree size and context length are read;
//    then warp 0 streams the K tiles of 128 keys and warp 3 the V tiles, each
//    through its own 2-slot ring with TMA (cp.async.bulk.tensor, 128-byte
//    swizzle, no multicast); a slot frees once both halves' MMAs have read it;
//  * the tile's keys are split into two halves of 64 that run as independent
//    pipelines, each with its own online softmax, TMEM buffers and MMA
//    issuer, so that one half's latency-bound phases (waiting for S, the TMEM
//    load, the max, handing P over) overlap the other half's exponentials;
//  * lane 0 of warp 1 + h issues half h's tcgen05.mma kind::f16 (bf16 in,
//    fp32 out): S_h = Q K_t[64 h : 64 h + 64]^T into one of its two TMEM
//    buffers (N = 64), issued as soon as the half's softmax has read the
//    buffer's previous tile, then O_h += P_h V_t[64 h : 64 h + 64] into its
//    accumulator (O_A at TMEM column 0, O_B at 384);
//  * warps 4-11 run the softmax, two warps per TMEM lane quadrant (one query
//    row per lane), warp 4 + 4 h for half h.  Each warp reads its S with
//    tcgen05.ld, applies the tree mask (context tiles are visible to every
//    row and skip it), and writes P_h as bf16 into shared memory in the MMA
//    operand layout; O_h is rescaled only when a row's running max grows by
//    more than 2^8 (the final normalisation uses the same reference max, so
//    this is exact).  Once every row has a reference, a fully visible tile is
//    exponentiated against it directly, its max taken alongside, and redone
//    the exact way only if some row grows;
//  * epilogue, after both halves' last PV: the pair exchanges its (max, sum)
//    once and writes (O_A 2^(m_A - M) + O_B 2^(m_B - M)) / l as bf16 (round to
//    nearest even).
// Every wait is bounded (~1 s); on a timeout the CTA flags the request, waits
// for its own copies and MMAs (bounded), frees its TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace bastion {

namespace {

constexpr int kAT = 384;  // warp 0 TMA (Q, K), 1-2 MMA (2 also TMEM), 3 TMA (V), 4-11 softmax
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr uint32_t kAtom = 128 * 128;          // 128 rows x 128 bytes
constexpr uint32_t kTile = 2 * kAtom;          // 128 x 128 bf16
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffKV = kTile;             // stage s: K at +0, V at +kTile
constexpr uint32_t kOffP = kOffKV + 2 * 2 * kTile;
constexpr uint32_t kOffBar = kOffP + 2 * kTile;
constexpr uint32_t kSmem = kOffBar + 256 + 1024;  // + alignment slack
constexpr float kRescale = 8.0f;               // lazy rescale threshold (log2 units)
constexpr uint32_t kColOB = 384;  // TMEM columns: O_A 0, S_A 128 and 192, S_B 256 and 320, O_B 384

struct AttnArgs {
  int B, n_max, Hq, Hkv, G, W, qt_max;
  int64_t L_cap;
  const int32_t *ctx_len, *n_nodes;
  const uint32_t *anc_mask;
  float scale_log2;
  uint16_t *out;
  int32_t *status;
};

struct Bars {
  // [h][s]: half h of the keys, buffer s
  uint64_t q_full, k_full[2], v_full[2], k_empty[2], v_empty[2], s_full[2][2], s_free[2][2],
      p_full[2][2], pv_done[2][2], mma_done[2];
  uint32_t tmem;
  int abort;
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// kind::f16 instruction descriptor: fp32 accumulate, bf16 A and B, M = 128, N = n.
__device__ __forceinline__ uint32_t idesc_bf16(bool b_mn_major, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}

__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// S = Q K^T for the keys whose rows start at sk (64 or 128 of them, as the
// instruction descriptor says): eight K = 16 steps over the two 64-column
// atoms of Q and K.
__device__ __forceinline__ void mma_qk(uint32_t d, uint32_t sq, uint32_t sk, uint32_t idesc) {
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    const uint32_t off = (uint32_t)(ks >> 2) * kAtom + (uint32_t)(ks & 3) * 32u;
    mma_bf16(d, sw128_desc(sq + off, 16, 1024), sw128_desc(sk + off, 16, 1024), idesc, ks > 0);
  }
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

// 64 consecutive columns of the warp's 32 lanes: two loads, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&v)[64]) {
  uint32_t r[64];
#pragma unroll
  for (int h = 0; h < 2; ++h)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
        "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[32 * h + 0]), "=r"(r[32 * h + 1]), "=r"(r[32 * h + 2]), "=r"(r[32 * h + 3]),
          "=r"(r[32 * h + 4]), "=r"(r[32 * h + 5]), "=r"(r[32 * h + 6]), "=r"(r[32 * h + 7]),
          "=r"(r[32 * h + 8]), "=r"(r[32 * h + 9]), "=r"(r[32 * h + 10]), "=r"(r[32 * h + 11]),
          "=r"(r[32 * h + 12]), "=r"(r[32 * h + 13]), "=r"(r[32 * h + 14]), "=r"(r[32 * h + 15]),
          "=r"(r[32 * h + 16]), "=r"(r[32 * h + 17]), "=r"(r[32 * h + 18]), "=r"(r[32 * h + 19]),
          "=r"(r[32 * h + 20]), "=r"(r[32 * h + 21]), "=r"(r[32 * h + 22]), "=r"(r[32 * h + 23]),
          "=r"(r[32 * h + 24]), "=r"(r[32 * h + 25]), "=r"(r[32 * h + 26]), "=r"(r[32 * h + 27]),
          "=r"(r[32 * h + 28]), "=r"(r[32 * h + 29]), "=r"(r[32 * h + 30]), "=r"(r[32 * h + 31])
        : "r"(taddr + 32u * (uint32_t)h));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// (x0, x1) * s + c, both lanes of a packed f32x2 FMA.
__device__ __forceinline__ void fma2(float x0, float x1, float sc, float c, float &d0, float &d1) {
  asm("{\n .reg .b64 x, m, a, d;\n mov.b64 x, {%2, %3};\n mov.b64 m, {%4, %4};\n"
      " mov.b64 a, {%5, %5};\n fma.rn.f32x2 d, x, m, a;\n mov.b64 {%0, %1}, d;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(x0), "f"(x1), "f"(sc), "f"(c));
}

__device__ __forceinline__ void add2(float &a0, float &a1, float b0, float b1) {
  asm("{\n .reg .b64 a, b;\n mov.b64 a, {%0, %1};\n mov.b64 b, {%2, %3};\n"
      " add.rn.f32x2 a, a, b;\n mov.b64 {%0, %1}, a;\n}\n"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Bounded wait that also honours the CTA's abort flag.
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

__device__ __forceinline__ uint32_t select_word(const uint32_t (&w)[8], int k) {
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) r = (k == i) ? w[i] : r;
  return r;
}

__global__ void __launch_bounds__(kAT, 1)
    tree_attention_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, AttnArgs a) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Bars &bs = *reinterpret_cast<Bars *>(smem + kOffBar);
  volatile int *abort = &bs.abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {  // the descriptors are parameters: fetch them while the producer kernel ends
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_v)) : "memory");
  }
  griddep_wait();
  griddep_launch_dependents();
  const int qt = blockIdx.x % a.qt_max;
  const int g = (blockIdx.x / a.qt_max) % a.Hkv;
  const int r = blockIdx.x / (a.qt_max * a.Hkv);
  const int nodes_per_tile = kBM / a.G;
  const int i0 = qt * nodes_per_tile;
  if (tid == 0) {
    mbar_init(&bs.q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bs.k_full[s], 1);
      mbar_init(&bs.v_full[s], 1);
      mbar_init(&bs.k_empty[s], 2);  // both halves' S MMAs have read the K slot
      mbar_init(&bs.v_empty[s], 2);  // both halves' PV MMAs have read the V slot
      for (int h = 0; h < 2; ++h) {
        mbar_init(&bs.s_full[h][s], 1);
        mbar_init(&bs.s_free[h][s], 4);
        mbar_init(&bs.p_full[h][s], 128);
        mbar_init(&bs.pv_done[h][s], 1);
      }
    }
    mbar_init(&bs.mma_done[0], 1);
    mbar_init(&bs.mma_done[1], 1);
    bs.abort = 0;
    fence_mbar_init();
    // Q and the first two K and V tiles start loading before anything else:
    // their coordinates depend on neither the tree's size nor the context
    // length (a tile past the cache reads the fill value); the producers
    // continue from tile 2
    mbar_arrive_expect_tx(&bs.q_full, kTile);
    tma_load_4d(smem + kOffQ, &tm_q, 0, g * a.G, i0, r, &bs.q_full);
    tma_load_4d(smem + kOffQ + kAtom, &tm_q, 64, g * a.G, i0, r, &bs.q_full);
    for (int t = 0; t < 2; ++t) {
      unsigned char *dk = smem + kOffKV + t * 2 * kTile;
      mbar_arrive_expect_tx(&bs.k_full[t], kTile);
      tma_load_4d(dk, &tm_k, 0, g, t * kBN, r, &bs.k_full[t]);
      tma_load_4d(dk + kAtom, &tm_k, 64, g, t * kBN, r, &bs.k_full[t]);
      mbar_arrive_expect_tx(&bs.v_full[t], kTile);
      tma_load_4d(dk + kTile, &tm_v, 0, g, t * kBN, r, &bs.v_full[t]);
      tma_load_4d(dk + kTile + kAtom, &tm_v, 64, g, t * kBN, r, &bs.v_full[t]);
    }
  }
  const int nn = a.n_nodes[r];
  const int ctx = a.ctx_len[r];
  const int rows = nn * a.G;
  if (nn < 1 || nn > a.n_max || qt * kBM >= rows) {
    if (tid == 0) {  // no rows here: the copies issued above land before the CTA leaves
      mbar_wait_bounded(&bs.q_full, 0);
      for (int t = 0; t < 2; ++t) {
        mbar_wait_bounded(&bs.k_full[t], 0);
        mbar_wait_bounded(&bs.v_full[t], 0);
      }
    }
    return;
  }
  int64_t keys = (int64_t)ctx + nn;
  if (ctx < 0 || keys > a.L_cap) {
    if (tid == 0 && qt == 0 && g == 0) atomicOr(&a.status[r], BASTION_STATUS_KV_OVERFLOW);
    keys = keys > a.L_cap ? a.L_cap : keys;
  }
  const int ctx_c = ctx < 0 ? 0 : ctx;
  const int n_tiles = (int)((keys + kBN - 1) / kBN);

  if (warp == 2) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(
                     smem_u32(&bs.tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bs.tmem;

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // warp 0: the K tiles from tile 2 on (a K slot frees once both halves'
    // S MMAs have read it); warp 3: the V tiles (a V slot frees once both
    // halves' PV MMAs have read it)
    if (lane == 0) {
      const bool is_k = warp == 0;
      uint64_t *full = is_k ? bs.k_full : bs.v_full, *empty = is_k ? bs.k_empty : bs.v_empty;
      const CUtensorMap *map = is_k ? &tm_k : &tm_v;
      int issued = 2;  // tiles 0 and 1 were issued at the start
      for (int t = 2; t < n_tiles; ++t) {
        const int s = t & 1;
        if (!wait_bar(&empty[s], ((t - 2) >> 1) & 1, abort, &a.status[r])) break;
        unsigned char *dst = smem + kOffKV + s * 2 * kTile + (is_k ? 0 : kTile);
        mbar_arrive_expect_tx(&full[s], kTile);
        tma_load_4d(dst, map, 0, g, t * kBN, r, &full[s]);
        tma_load_4d(dst + kAtom, map, 64, g, t * kBN, r, &full[s]);
        issued = t + 1;
      }
      // drain: our last copies have landed (bounded) before the CTA may exit
      for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t)
        mbar_wait_bounded(&full[t & 1], (t >> 1) & 1);
      if (is_k) mbar_wait_bounded(&bs.q_full, 0);
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // lane 0 of warp 1 + h issues half h's MMAs: S_h = Q K^T over keys
    // [64 h, 64 h + 64) of each tile into its own two TMEM buffers, and
    // O_h += P_h V over the same keys.  The halves are independent pipelines:
    // neither waits for the other's softmax, so one half's latency-bound
    // phases overlap the other's exponentials.
    const int h = warp - 1;
    if (lane == 0) {
      const uint32_t id_qk = idesc_bf16(false, 64), id_pv = idesc_bf16(true, 128);
      const uint32_t sq = smem_u32(smem + kOffQ);
      const uint32_t s_col = tmem + 128u + 128u * (uint32_t)h;  // S_h buffer s at + 64 s
      const uint32_t o_col = tmem + (h ? kColOB : 0u);
      bool ok = wait_bar(&bs.q_full, 0, abort, &a.status[r]);
      tc_fence_after();
      // S_0 and S_1 first; then, per tile u, S_{u+2} goes into buffer u % 2
      // as soon as the half's softmax warps have read S_u, ahead of
      // O_h += P_u V_u, so the softmax never finds its S queued behind a PV
      for (int t = 0; ok && t < n_tiles && t < 2; ++t) {
        if (!wait_bar(&bs.k_full[t], 0, abort, &a.status[r])) ok = false;
        if (!ok) break;
        tc_fence_after();
        mma_qk(s_col + 64u * (uint32_t)t, sq, smem_u32(smem + kOffKV + t * 2 * kTile) + 8192u * (uint32_t)h,
               id_qk);
        mma_commit(&bs.s_full[h][t]);
        mma_commit(&bs.k_empty[t]);
      }
      for (int u = 0; ok && u < n_tiles; ++u) {
        const int s = u & 1;
        if (u + 2 < n_tiles) {
          if (!wait_bar(&bs.s_free[h][s], (u >> 1) & 1, abort, &a.status[r])) break;
          if (!wait_bar(&bs.k_full[s], ((u + 2) >> 1) & 1, abort, &a.status[r])) break;
          tc_fence_after();
          mma_qk(s_col + 64u * (uint32_t)s, sq, smem_u32(smem + kOffKV + s * 2 * kTile) + 8192u * (uint32_t)h,
                 id_qk);
          mma_commit(&bs.s_full[h][s]);
          mma_commit(&bs.k_empty[s]);
        }
        if (!wait_bar(&bs.p_full[h][s], (u >> 1) & 1, abort, &a.status[r])) break;
        if (!wait_bar(&bs.v_full[s], (u >> 1) & 1, abort, &a.status[r])) break;
        tc_fence_after();
        // P_h is atom h of P buffer s; V rows 64 h .. 64 h + 63 of slot s
        const uint32_t sp = smem_u32(smem + kOffP + s * kTile) + (uint32_t)h * kAtom;
        const uint32_t sv = smem_u32(smem + kOffKV + s * 2 * kTile + kTile) + 8192u * (uint32_t)h;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(o_col, sw128_desc(sp + (uint32_t)ks * 32u, 16, 1024),
                   sw128_desc(sv + (uint32_t)ks * 2048u, kAtom, 1024), id_pv, (u > 0 || ks > 0));
        mma_commit(&bs.pv_done[h][s]);
        mma_commit(&bs.v_empty[s]);
      }
      // every MMA this thread issued has completed (bounded) before the CTA
      // may free its TMEM
      mma_commit(&bs.mma_done[h]);
      mbar_wait_bounded(&bs.mma_done[h], 0);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax + epilogue
    // warps w and w + 4 (w = 4..7) share TMEM lane quadrant w - 4: the same 32
    // query rows.  Half h takes keys [64 h, 64 h + 64) of every tile with its
    // own online softmax (reference max, sum) and its own accumulator O_h;
    // the two halves are combined once, at the end.
    const int quad = (warp - 4) & 3, half = (warp - 4) >> 2;
    const int m = quad * 32 + lane;  // query row = TMEM lane
    const int node = i0 + m / a.G;
    const int hh = m % a.G;
    const bool row_live = node < nn;
    uint32_t anc[8];
#pragma unroll
    for (int w = 0; w < 8; ++w)
      anc[w] = (row_live && w < a.W) ? a.anc_mask[((size_t)r * a.n_max + node) * a.W + w] : 0u;
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    const uint32_t col0 = 64u * (uint32_t)half;
    const uint32_t o_base = lane_base + (half ? kColOB : 0u);
    float m_ref = -INFINITY, l_sum = 0.f;
    bool all_ref = false;  // every row of the warp has a reference max
    bool ok = true;
    for (int t = 0; t < n_tiles && ok; ++t) {
      const int s = t & 1;
      ok = __all_sync(kFull, wait_bar(&bs.s_full[half][s], (t >> 1) & 1, abort, &a.status[r]));
      if (!ok) break;
      tc_fence_after();
      const int kb = t * kBN + 64 * half;
      // visibility of this half's 64 keys, 32 per word
      uint32_t vis[2] = {0xffffffffu, 0xffffffffu};
      const bool ctx_tile = kb + 64 <= ctx_c;  // the context: visible to every row
#pragma unroll
      for (int q = 0; q < 2 && !ctx_tile; ++q) {
        const int j0 = kb + 32 * q;           // first key of the group
        uint32_t ctxbits;
        if (j0 + 32 <= ctx_c) ctxbits = 0xffffffffu;
        else if (j0 >= ctx_c) ctxbits = 0u;
        else ctxbits = (1u << (ctx_c - j0)) - 1u;
        const int t0 = j0 - ctx_c;            // tree index of the first key
        uint32_t tb = 0u;
        if (t0 + 32 > 0 && t0 < 256) {
          if (t0 >= 0) {
            const int w0 = t0 >> 5, sh = t0 & 31;
            tb = select_word(anc, w0) >> sh;
            if (sh) tb |= select_word(anc, w0 + 1) << (32 - sh);
          } else {
            tb = select_word(anc, 0) << (-t0);
          }
        }
        uint32_t lim = 0xffffffffu;  // keys at or past the end are never visible
        const int64_t left = keys - j0;
        if (left <= 0) lim = 0u;
        else if (left < 32) lim = (1u << left) - 1u;
        vis[q] = (ctxbits | tb) & lim;
      }
      // this half's raw scores and the max of the visible ones, scaled (the
      // scale is positive); context tiles are fully visible to every row
      const bool full = __all_sync(kFull, (vis[0] & vis[1]) == 0xffffffffu);
      float v[64];
      const uint32_t s_addr = lane_base + 128u + 128u * (uint32_t)half + 64u * (uint32_t)s;
      tmem_ld64(s_addr, v);
      // At most two passes.  Once every row has a reference max, a fully
      // visible tile is first exponentiated against the current references,
      // its max taken alongside; only if some row's tile max exceeds its
      // reference by more than 2^8 is the tile redone the exact way (max
      // first, then the lazy rescale), which gives the same values whenever
      // no row grows, so the max leaves the critical path of the common tile.
      bool spec = full && all_ref, redo = false;
      bool p_free = t < 2;
      float part = 0.f;
      for (;;) {
        if (!spec) {
          if (redo) tmem_ld64(s_addr, v);  // the speculative pass consumed v
          float mr = -INFINITY;
          if (full) {
            float q0 = v[0], q1 = v[1], q2 = v[2], q3 = v[3];
#pragma unroll
            for (int i = 4; i < 64; i += 8) {
              q0 = max3f(q0, v[i], v[i + 1]);
              q1 = max3f(q1, v[i + 2], v[i + 3]);
              q2 = max3f(q2, v[i + 4], v[i + 5]);
              q3 = max3f(q3, v[i + 6], v[i + 7]);
            }
            mr = max3f(fmaxf(q0, q1), q2, q3);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if ((vis[0] >> i) & 1u) mr = fmaxf(mr, v[i]);
              if ((vis[1] >> i) & 1u) mr = fmaxf(mr, v[32 + i]);
            }
          }
          const float mt = mr * a.scale_log2;
          // lazy rescale: a row moves its reference max only when the tile
          // max exceeds it by more than 2^8; O_h in TMEM is rescaled by the
          // whole warp (tcgen05.ld/st are warp-collective), with alpha = 1 for
          // other rows.
          const bool grow = mt > m_ref + kRescale || (m_ref == -INFINITY && mt != -INFINITY);
          const bool rescale = grow && t > 0 && m_ref != -INFINITY;
          const float alpha = rescale ? ex2f(m_ref - mt) : 1.0f;
          if (__any_sync(kFull, rescale)) {
            ok = __all_sync(kFull, wait_bar(&bs.pv_done[half][(t - 1) & 1], ((t - 1) >> 1) & 1, abort,
                                            &a.status[r]));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
              float o[32];
              tmem_ld32(o_base + 32u * cc, o);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[i] *= alpha;
              tmem_st32(o_base + 32u * cc, o);
            }
          }
          if (rescale) l_sum *= alpha;
          if (grow) m_ref = mt;
          all_ref = __all_sync(kFull, m_ref != -INFINITY);
        }
        if (!p_free) {  // P buffer s free: PV of tile t-2 done
          ok = __all_sync(kFull, wait_bar(&bs.pv_done[half][s], ((t - 2) >> 1) & 1, abort, &a.status[r]));
          if (!ok) break;
          p_free = true;
        }
        unsigned char *pb = smem + kOffP + s * kTile;
        part = 0.f;
        float mx[2] = {-INFINITY, -INFINITY};
        const float nm = m_ref == -INFINITY ? 0.f : -m_ref;  // no visible key yet: all p = 0
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t pk[16];
          if (full && m_ref != -INFINITY) {
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float t0, t1;
              fma2(v[32 * cc + i], v[32 * cc + i + 1], a.scale_log2, nm, t0, t1);
              const float p0 = ex2f(t0), p1 = ex2f(t1);
              mx[cc] = max3f(mx[cc], v[32 * cc + i], v[32 * cc + i + 1]);
              add2(s0, s1, p0, p1);
              pk[i >> 1] = pack_bf16(p0, p1);
            }
            part += s0 + s1;
          } else {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const bool s0 = ((vis[cc] >> i) & 1u) && m_ref != -INFINITY;
              const bool s1 = ((vis[cc] >> (i + 1)) & 1u) && m_ref != -INFINITY;
              const float p0 = s0 ? ex2f(fmaf(v[32 * cc + i], a.scale_log2, nm)) : 0.f;
              const float p1 = s1 ? ex2f(fmaf(v[32 * cc + i + 1], a.scale_log2, nm)) : 0.f;
              part += p0 + p1;
              pk[i >> 1] = pack_bf16(p0, p1);
            }
          }
          // columns 64 h + 32 cc ..: atom h, 16-byte chunks (4 cc + q) ^ (m % 8)
          unsigned char *rowp = pb + half * kAtom + (m >> 3) * 1024 + (m & 7) * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int ch = (cc * 4 + q) ^ (m & 7);
            *reinterpret_cast<uint4 *>(rowp + ch * 16) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (spec && __any_sync(kFull, fmaxf(mx[0], mx[1]) * a.scale_log2 > m_ref + kRescale)) {
          spec = false;  // some row grows: redo the tile exactly
          redo = true;
          continue;
        }
        break;
      }
      // S_t is no longer needed: its TMEM buffer may take S_{t+2} (a failed
      // warp releases it too, so the issuer is never left waiting on it)
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bs.s_free[half][s]);
      if (!ok) break;
      l_sum += part;
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&bs.p_full[half][s]);
    }
    // epilogue: the pair exchanges (reference max, sum) once -- both warps
    // always reach this barrier, a failed one with a NaN -- and each warp
    // writes its half of the columns: O = (O_A 2^(m_A - M) + O_B 2^(m_B - M)) /
    // (l_A 2^(m_A - M) + l_B 2^(m_B - M)), M = max(m_A, m_B).
    if (n_tiles > 0) {
      bool okw = ok;
      if (okw) {
        const int u = n_tiles - 1;
        okw = __all_sync(kFull, wait_bar(&bs.pv_done[half][u & 1], (u >> 1) & 1, abort, &a.status[r]));
      }
      // both halves' last PV has completed (every softmax warp passes its own
      // wait, or fails it, before this barrier): P buffer 0 is free and O_A,
      // O_B are final
      tc_fence_before();
      asm volatile("bar.sync 5, 256;" ::: "memory");
      tc_fence_after();
      // the exchange uses P buffer 0: the last PV has read it (a warp that
      // failed only writes its NaN flag)
      float *xm = reinterpret_cast<float *>(smem + kOffP);  // [2][128] maxima
      float *xl = xm + 256;                                  // [2][128] sums
      xm[half * 128 + m] = okw ? m_ref : __int_as_float(0x7fc00001);
      xl[half * 128 + m] = l_sum;
      asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
      const float mA = xm[m], mB = xm[128 + m], lA = xl[m], lB = xl[128 + m];
      ok = __all_sync(kFull, !(mA != mA) && !(mB != mB));
      if (ok) {
        const float M = fmaxf(mA, mB);
        const float fA = mA == -INFINITY ? 0.f : ex2f(mA - M);
        const float fB = mB == -INFINITY ? 0.f : ex2f(mB - M);
        const float l = lA * fA + lB * fB;
        const float inv = row_live && l > 0.f ? 1.0f / l : 0.0f;
        const float gA = fA * inv, gB = fB * inv;
        uint16_t *dst = a.out + (((size_t)r * a.n_max + (row_live ? node : 0)) * a.Hq +
                                 (size_t)g * a.G + hh) * 128 + col0;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float oa[32], ob[32];
          tmem_ld32(lane_base + col0 + 32u * cc, oa);
          tmem_ld32(lane_base + kColOB + col0 + 32u * cc, ob);
          if (row_live) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 pkt;
              pkt.x = pack_bf16(oa[8 * q + 0] * gA + ob[8 * q + 0] * gB, oa[8 * q + 1] * gA + ob[8 * q + 1] * gB);
              pkt.y = pack_bf16(oa[8 * q + 2] * gA + ob[8 * q + 2] * gB, oa[8 * q + 3] * gA + ob[8 * q + 3] * gB);
              pkt.z = pack_bf16(oa[8 * q + 4] * gA + ob[8 * q + 4] * gB, oa[8 * q + 5] * gA + ob[8 * q + 5] * gB);
              pkt.w = pack_bf16(oa[8 * q + 6] * gA + ob[8 * q + 6] * gB, oa[8 * q + 7] * gA + ob[8 * q + 7] * gB);
              *reinterpret_cast<uint4 *>(dst + 32 * cc + 8 * q) = pkt;
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// The driver's tensor-map encoder, looked up once (a function-local static:
// its initialisation is thread-safe, so concurrent first calls are too).
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

bool make_map(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
              uint32_t b0, uint32_t b1, uint32_t b2) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  cuuint32_t box[4] = {b0, b1, b2, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult rc = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides,
                    box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return rc == CUDA_SUCCESS;
}

}  // namespace

size_t attention_workspace_bytes(int, int, int, int, int, int64_t) { return 256; }

int launch_attention(const void *q, const void *k, const void *v, int B, int n_max, int Hq,
                     int Hkv, int D, int64_t L_cap, const int32_t *ctx_len,
                     const int32_t *n_nodes, const uint32_t *anc_mask, float scale, void *out,
                     void *ws, int32_t *status, cudaStream_t stream) {
  (void)ws;
  (void)D;
  const int G = Hq / Hkv;
  if (128 % G) return BASTION_ERR_UNSUPPORTED;
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, q, 128, (uint64_t)Hq, (uint64_t)n_max, (uint64_t)B, 64, (uint32_t)G,
                (uint32_t)(128 / G)) ||
      !make_map(&mk, k, 128, (uint64_t)Hkv, (uint64_t)L_cap, (uint64_t)B, 64, 1, 128) ||
      !make_map(&mv, v, 128, (uint64_t)Hkv, (uint64_t)L_cap, (uint64_t)B, 64, 1, 128))
    return BASTION_ERR_LAUNCH;
  AttnArgs a;
  a.B = B;
  a.n_max = n_max;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.G = G;
  a.W = (n_max + 31) / 32;
  a.qt_max = (n_max * G + kBM - 1) / kBM;
  a.L_cap = L_cap;
  a.ctx_len = ctx_len;
  a.n_nodes = n_nodes;
  a.anc_mask = anc_mask;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = static_cast<uint16_t *>(out);
  a.status = status;
  cudaFuncSetAttribute(tree_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  const long long grid = (long long)B * Hkv * a.qt_max;
  const cudaError_t e = launch_pdl(tree_attention_kernel, dim3((unsigned)grid), dim3(kAT), kSmem,
                                   stream, mq, mk, mv, a);
  return (e == cudaSuccess && cudaGetLastError() == cudaSuccess) ? BASTION_OK : BASTION_ERR_LAUNCH;
}

}  // namespace bastion
