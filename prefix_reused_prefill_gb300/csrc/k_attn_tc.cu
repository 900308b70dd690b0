// Causal grouped-query attention for many new rows on the 5th-generation
// tensor cores: S = Q K^T and P V as tcgen05.mma with accumulators in TMEM.
//
// goinfer, "Turn nine in under half a second" ("What goinfer does"): the 254
// new rows of turn 9 attend to the 1668 cached rows plus themselves; with
// all G query heads of a KV head packed as rows (row = token*G + head in the
// group), one KV head's rows form a real dense contraction.
//
// One CTA = (128-row tile of one KV head, key split); keys go in blocks of
// 128, so S_j = Q K_j^T is M=128, N=128 (the MMA count of a block, not its
// size, bounds a small-tile tensor pipe).  Tensor memory holds three S
// buffers of 128 columns and the O accumulator (512 columns).  Warp roles:
//   warp 0     TMA, two independent streams: lane 0 the Q tile once (128 rows x
//              d, 128B-swizzled K-major) and per block a K tile ([128 keys][d],
//              3 stages, a stage freed by the S that read it), lane 1 per block
//              a V^T tile ([d][128 keys]; V is stored transposed in the slot; 2
//              stages, freed by the P V that read it);
//   warp 1     allocates TMEM; one thread issues S_j into S buffer j % 3 as
//              soon as its K tile is in and P V of the buffer's previous block
//              has completed;
//   warp 10    one thread issues O += P_j V_j (M=128, N=d) with P_j read from
//              tensor memory, in block order;
//   warps 2-9  two threads per row, one per 64-key half of the block (warps
//              w and w+4 share a TMEM lane quarter): tcgen05.ld of their half of
//              S_j, causal mask, the block max exchanged through shared memory
//              (a named barrier per warp pair), online softmax in fp32 (log2
//              units), and P_j (bf16) stored back over the first half of its own
//              S buffer with tcgen05.st.  Each thread keeps the running sum of
//              its half; the halves are added at the end.  The running-max
//              correction of O is lazy: P_j is taken relative to a per-row
//              reference max, and only when a block's max exceeds the reference
//              by more than 8 (P would exceed 2^8) do the two threads rescale
//              their halves of the row of O in TMEM (after P V of the previous
//              block) and move the reference.  At the end O / l is written (or,
//              with several key splits, the unnormalised partials merged by
//              attn_combine).
// Every wait is bounded; a timed-out CTA records it, drains its copies and
// frees its TMEM.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kKeys = kAttnTcKeys;               // 128 keys per block
constexpr int kSoftmaxWarps = 8;                  // warps 2..9
constexpr int kPvWarp = 2 + kSoftmaxWarps;        // warp 10
constexpr int kThreads = 32 * (kPvWarp + 1);

template <int D>
struct TcCfg {
  static constexpr int kQBytes = 128 * D * 2;    // D/64 atoms of [128 rows][64 elems]
  static constexpr int kKAtom = kKeys * 128;     // [128 keys][64 elems]
  static constexpr int kKBytes = kKeys * D * 2;  // D/64 atoms
  static constexpr int kVAtom = D * 128;         // [D rows][64 keys]
  static constexpr int kVBytes = D * kKeys * 2;  // 2 atoms
  static constexpr int kKStages = 3;
  static constexpr int kVStages = 2;
  static constexpr int kSmem = kQBytes + kKStages * kKBytes + kVStages * kVBytes + 1024;
  // TMEM columns: S (then P) buffers at 0, 128, 256; the O accumulator at 384
  static constexpr int kSBufs = 3;
  static __device__ __forceinline__ uint32_t scol(int b) { return (uint32_t)(128 * b); }
  static constexpr uint32_t kOCol = 384;
  static constexpr int kTmemCols = 512;
  static_assert(128 * (D + 4) * 4 <= kKStages * kKBytes, "the O tile fits the K ring");
};

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
__device__ __forceinline__ uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (TMEM) += A (TMEM) * B (shared memory)
__device__ __forceinline__ void mma_f16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
// 2^x with the PTX approximate base-2 exponential (ex2.approx.ftz.f32; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLazyMax = 8.0f;  // rescale O only when a block max passes the reference by this (log2)

// tcgen05.ld without the wait (several loads in flight, then tmem_wait_ld)
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t r[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t r[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float v[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnParams p) {
  using C = TcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t q_full;
  __shared__ __align__(8) uint64_t k_full[C::kKStages], k_empty[C::kKStages];
  __shared__ __align__(8) uint64_t v_full[C::kVStages], v_empty[C::kVStages];
  __shared__ __align__(8) uint64_t s_full[C::kSBufs], p_full[C::kSBufs], pv_done[C::kSBufs];
  __shared__ float xmax[2][2][128];   // [block parity][key half][row]
  __shared__ float xsum[2][128];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t q_base = base;
  const uint32_t k_base = q_base + C::kQBytes;
  const uint32_t v_base = k_base + C::kKStages * C::kKBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rt = blockIdx.x, split = blockIdx.y, kv = blockIdx.z;
  const int R = p.G * p.rows.m;
  const int row_lo = rt * 128;
  const int row_hi = min(R, row_lo + 128);
  const int last_tok = (row_hi - 1) / p.G;
  const int kend = p.rows.P + last_tok + 1;
  const int nb = (kend + kKeys - 1) / kKeys;
  const int b0 = (int)((long long)nb * split / p.nsplit);
  const int b1 = (int)((long long)nb * (split + 1) / p.nsplit);
  const int nblk = b1 - b0;

  dev::pdl_trigger();
  if (threadIdx.x == 0) {
    dev::mbar_init(dev::smem_u32(&q_full), 1);
    for (int i = 0; i < C::kKStages; ++i) {
      dev::mbar_init(dev::smem_u32(&k_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&k_empty[i]), 1);
    }
    for (int i = 0; i < C::kVStages; ++i) {
      dev::mbar_init(dev::smem_u32(&v_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&v_empty[i]), 1);
    }
    for (int i = 0; i < C::kSBufs; ++i) {
      dev::mbar_init(dev::smem_u32(&s_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&p_full[i]), kSoftmaxWarps);
      dev::mbar_init(dev::smem_u32(&pv_done[i]), 1);
    }
    // a wait has given up earlier in the call: the CTA issues no copy and
    // runs no role (one decision for the whole CTA, read after the
    // allocation's barrier rather than behind a barrier of its own)
    *abort_v = dev::status_set(p.status) ? 1 : 0;
    dev::fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dev::smem_u32(&tmem_slot)),
                 "r"(C::kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (*abort_v) goto teardown;
  // q and this call's K/V come from the previous launch; only the producers'
  // loads of cached-prefix K/V may run ahead of it.
  if (warp != 0 || lane > 1) dev::pdl_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- producers
    if (lane <= 1 && nblk == 0) dev::pdl_wait();
    if (lane <= 1 && nblk > 0) {
      const bool is_k = lane == 0;
      const int stages = is_k ? C::kKStages : C::kVStages;
      dev::prefetch_tmap(is_k ? &p.tkv : &p.tvt);
      if (is_k) dev::prefetch_tmap(&p.tq);
      uint64_t* fullb = is_k ? k_full : v_full;
      uint64_t* emptyb = is_k ? k_empty : v_empty;
      const uint32_t ring = is_k ? k_base : v_base;
      const uint32_t bytes = is_k ? C::kKBytes : C::kVBytes;
      // a block = two 64-key halves: K atoms of 128 rows (two 64-row boxes each),
      // V^T atoms of 64 keys
      auto load = [&](int j, uint32_t dst, uint32_t fb) {
        const int key0 = (b0 + j) * kKeys;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (is_k) {
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
              dev::tma_load_2d(dst + a * C::kKAtom + h * (64 * 128), &p.tkv, 64 * a,
                               p.kbase + kv * p.cap + key0 + 64 * h, fb);
          } else {
            dev::tma_load_2d(dst + h * C::kVAtom, &p.tvt, key0 + 64 * h, p.vtbase + kv * D, fb);
          }
        }
      };
      auto prefetch = [&](int j) {
        const int key0 = (b0 + j) * kKeys;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if (is_k) {
#pragma unroll
            for (int a = 0; a < D / 64; ++a)
              dev::tma_prefetch_2d(&p.tkv, 64 * a, p.kbase + kv * p.cap + key0 + 64 * h);
          } else {
            dev::tma_prefetch_2d(&p.tvt, key0 + 64 * h, p.vtbase + kv * D);
          }
        }
      };
      int pre = 0;
      while (pre < nblk && pre < stages && (b0 + pre + 1) * kKeys <= p.rows.P) {
        const uint32_t fb = dev::smem_u32(&fullb[pre]);
        dev::mbar_arrive_expect_tx(fb, bytes);
        load(pre, ring + pre * bytes, fb);
        ++pre;
      }
      // the rest of the cached-prefix blocks of this split toward L2
      for (int j = pre; j < nblk && (b0 + j + 1) * kKeys <= p.rows.P; ++j) prefetch(j);
      dev::pdl_wait();
      const uint32_t qb = dev::smem_u32(&q_full);
      if (is_k) {
        dev::mbar_arrive_expect_tx(qb, C::kQBytes);
        const int qrow = p.qrow0 + kv * R + row_lo;
#pragma unroll
        for (int a = 0; a < D / 64; ++a) dev::tma_load_2d(q_base + a * 16384, &p.tq, 64 * a, qrow, qb);
      }
      int issued = pre;
      for (int j = pre; j < nblk; ++j) {
        const int st = j % stages;
        if (j >= stages &&
            (!dev::mbar_wait(dev::smem_u32(&emptyb[st]), ((j / stages) - 1) & 1, p.status) || *abort_v)) {
          *abort_v = 1;
          break;
        }
        const uint32_t fb = dev::smem_u32(&fullb[st]);
        dev::mbar_arrive_expect_tx(fb, bytes);
        load(j, ring + st * bytes, fb);
        ++issued;
      }
      const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
      if (is_k) dev::mbar_wait_until(qb, 0, deadline);
      for (int st = 0; st < stages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / stages) * stages + st;
        dev::mbar_wait_until(dev::smem_u32(&fullb[st]), (uint32_t)(last / stages) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- S issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t id_qk = idesc_bf16(128, kKeys);
      bool ok = dev::mbar_wait(dev::smem_u32(&q_full), 0, p.status);
      const uint64_t qd = sw128_desc(q_base);
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j % C::kKStages, sb = j % C::kSBufs;
        if (!dev::mbar_wait(dev::smem_u32(&k_full[st]), (j / C::kKStages) & 1, p.status) ||
            (j >= C::kSBufs &&
             !dev::mbar_wait(dev::smem_u32(&pv_done[sb]), ((j / C::kSBufs) - 1) & 1, p.status)) ||
            *abort_v) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = sw128_desc(k_base + st * C::kKBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16(tmem + C::scol(sb), qd + (kk >> 2) * (16384 >> 4) + 2 * (kk & 3),
                  kd + (kk >> 2) * (C::kKAtom >> 4) + 2 * (kk & 3), id_qk, kk > 0 ? 1u : 0u);
        mma_commit(dev::smem_u32(&s_full[sb]));
        mma_commit(dev::smem_u32(&k_empty[st]));
      }
      if (!ok) *abort_v = 1;
    }
  } else if (warp == kPvWarp) {
    // ---------------------------------------------------------------- P V issuer
    // O += P_j V_j in block order, P_j from tensor memory; the commit frees
    // the V stage and, for the S issuer, the S / P buffer
    if (lane == 0 && nblk > 0) {
      const uint32_t id_pv = idesc_bf16(128, D);
      bool ok = true;
      for (int b = 0; b < nblk && ok; ++b) {
        const int st = b % C::kVStages, sb = b % C::kSBufs;
        if (!dev::mbar_wait(dev::smem_u32(&v_full[st]), (b / C::kVStages) & 1, p.status) ||
            !dev::mbar_wait(dev::smem_u32(&p_full[sb]), (b / C::kSBufs) & 1, p.status) || *abort_v) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t vd = sw128_desc(v_base + st * C::kVBytes);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_f16_ta(tmem + C::kOCol, tmem + C::scol(sb) + 8u * (uint32_t)kk,
                     vd + (kk >> 2) * (C::kVAtom >> 4) + 2 * (kk & 3), id_pv, (b > 0 || kk > 0) ? 1u : 0u);
        mma_commit(dev::smem_u32(&pv_done[sb]));
        mma_commit(dev::smem_u32(&v_empty[st]));
      }
      if (!ok) *abort_v = 1;
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int q4 = warp & 3;                  // TMEM lane quarter
    const int half = (warp - 2) >> 2;         // keys [64 half, 64 half + 64) of each block
    const int r = 32 * q4 + lane;
    const uint32_t tlane = (uint32_t)(32 * q4) << 16;
    const int pair_bar = 1 + q4;              // warps q4+2 and q4+6 (64 threads)
    const int rho = row_lo + r;
    int tok = -1, head = 0, lo = 1, hi = 0;
    if (rho < R) {
      tok = rho / p.G;
      head = kv * p.G + rho % p.G;
      const int br = row_branch(p.rows, tok);
      lo = p.rows.P + p.rows.off[br];
      hi = p.rows.P + tok;
    }
    const int P0 = p.rows.P;
    float m_ref = -INFINITY, l = 0.f;
    // warp-uniform; once false the warp skips work and waits but still meets
    // its partner at every pair barrier
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int xb = j & 1;                // exchange slot
      const int sb = j % C::kSBufs;        // S / P buffer
      if (ok) {
        const bool got = dev::mbar_wait(dev::smem_u32(&s_full[sb]), (j / C::kSBufs) & 1, p.status) && !*abort_v;
        ok = __all_sync(0xffffffffu, got);
      }
      float sv[64];
      float mx = -INFINITY;
      const int key0 = (b0 + j) * kKeys + 64 * half;
      if (ok) {
        tc_fence_after();
        uint32_t sr[64];
        tmem_ld32_nowait(tmem + tlane + C::scol(sb) + 64 * half, sr);
        tmem_ld32_nowait(tmem + tlane + C::scol(sb) + 64 * half + 32, sr + 32);
        tmem_wait_ld();
        // visible keys of this row within the half block: [0, P) and [lo, hi]
        const int pe = min(max(P0 - key0, 0), 64);
        const int la = min(max(lo - key0, 0), 64);
        const int hb = tok >= 0 ? min(max(hi - key0 + 1, 0), 64) : 0;
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        // raw scores here; the log2-domain scale is applied inside the
        // exponent's FMA below (the scale is positive, so the max commutes)
        if (pe == 64) {
          // wholly inside the cached prefix: every key visible.  (pe is the same
          // for every row, so the warp takes one path; a row past the tile's
          // last token keeps its scores but a block max of -inf, so its O row,
          // never stored, moves no reference and rescales nothing.)
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            sv[k] = __uint_as_float(sr[k]);
            m4[k & 3] = fmaxf(m4[k & 3], sv[k]);
          }
          if (tok < 0) m4[0] = m4[1] = m4[2] = m4[3] = -INFINITY;
        } else {
#pragma unroll
          for (int k = 0; k < 64; ++k) {
            const bool vis = tok >= 0 && (k < pe || (k >= la && k < hb));
            sv[k] = vis ? __uint_as_float(sr[k]) : -INFINITY;
            m4[k & 3] = fmaxf(m4[k & 3], sv[k]);
          }
        }
        mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
      }
      // the row's block max from both halves; after this barrier both halves
      // have read their S, so P may overwrite the buffer
      xmax[xb][half][r] = mx;
      named_sync(pair_bar, 64);
      mx = fmaxf(mx, xmax[xb][half ^ 1][r]);
      if (!ok) continue;
      // lazy reference max: move it (and rescale O) only when P would exceed 2^8
      const bool move = mx > m_ref + kLazyMax;
      const float m_new = move ? mx : m_ref;
      const float factor = (move && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
      const float muse = m_new == -INFINITY ? 0.f : m_new;
      uint32_t pk[32];
      float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 64; k += 2) {
        const float e0 = ex2_approx(fmaf(sv[k], p.scale_log2, -muse));
        const float e1 = ex2_approx(fmaf(sv[k + 1], p.scale_log2, -muse));
        s4[(k >> 1) & 3] += e0 + e1;
        pk[k / 2] = dev::pack_bf16x2(e0, e1);
      }
      const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
      // P_j (bf16, keys in order, two per column) over the first half of S_j
      tmem_st32(tmem + tlane + C::scol(sb) + 32 * half, pk);
      // an O rescale waits for P V of the previous block
      const bool rescale = j >= 1 && __any_sync(0xffffffffu, factor != 1.f);
      if (rescale) {
        const bool got = dev::mbar_wait(dev::smem_u32(&pv_done[(j - 1) % C::kSBufs]),
                                        ((j - 1) / C::kSBufs) & 1, p.status);
        ok = __all_sync(0xffffffffu, got && !*abort_v);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t v[32];
            const uint32_t oaddr = tmem + tlane + C::kOCol + (D / 2) * half + c0;
            tmem_ld32_nowait(oaddr, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * factor);
            tmem_st32(oaddr, v);
          }
        }
      }
      tmem_wait_st();
      l = l * factor + sum;
      m_ref = m_new;
      tc_fence_before();
      __syncwarp();
      if (ok && lane == 0) dev::mbar_arrive(dev::smem_u32(&p_full[sb]));
    }
    if (ok && nblk > 0) {
      const bool got = dev::mbar_wait(dev::smem_u32(&pv_done[(nblk - 1) % C::kSBufs]),
                                      ((nblk - 1) / C::kSBufs) & 1, p.status) && !*abort_v;
      ok = __all_sync(0xffffffffu, got);
    }
    if (!ok) *abort_v = 1;
    // the row sum from both halves
    xsum[half][r] = l;
    named_sync(pair_bar, 64);
    l += xsum[half ^ 1][r];
    // O (divided by l with one key split; the unnormalised partial with
    // several) through shared memory, so that the stores to global memory go
    // a whole row per warp instruction: [128 rows][kOStride floats] over the K
    // ring, which the last S product has finished reading (the last P V is
    // complete, and the tensor core completes its products in order).  The
    // stride keeps both the row-wise v4 writes and the row reads conflict-free.
    constexpr int kOStride = D + 4;
    float* ost = reinterpret_cast<float*>(smem_raw + (k_base - dev::smem_u32(smem_raw)));
    if (ok) {
      tc_fence_after();
      const float sc = p.nsplit == 1 ? (l > 0.f ? 1.f / l : 0.f) : 1.f;
#pragma unroll
      for (int c0 = (D / 2) * half; c0 < (D / 2) * (half + 1); c0 += 32) {
        float v[32];
        if (nblk > 0) {
          tmem_ld32(tmem + tlane + C::kOCol + c0, v);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          *reinterpret_cast<float4*>(ost + r * kOStride + c0 + 4 * c4) =
              make_float4(v[4 * c4] * sc, v[4 * c4 + 1] * sc, v[4 * c4 + 2] * sc, v[4 * c4 + 3] * sc);
      }
      if (tok >= 0 && p.nsplit > 1 && half == 0) {
        const long long plane = (long long)p.rows.m * p.Hq;
        p.ml[split * plane + (long long)tok * p.Hq + head] = make_float2(m_ref, l);
      }
    }
    named_sync(5, 32 * kSoftmaxWarps);
    if (ok) {
      // warp w of the softmax warps writes rows 16 w .. 16 w + 15, a lane per
      // four head dims
      const int sw = warp - 2;
      const long long plane = (long long)p.rows.m * p.Hq;
      for (int rr = 16 * sw; rr < 16 * sw + 16; ++rr) {
        const int rho2 = row_lo + rr;
        if (rho2 >= R) break;
        const int tk = rho2 / p.G, hd = kv * p.G + rho2 % p.G;
        const long long ridx = (long long)tk * p.Hq + hd;
        for (int c = 4 * lane; c < D; c += 128) {
          const float4 x = *reinterpret_cast<const float4*>(ost + rr * kOStride + c);
          if (p.nsplit == 1) {
            uint2 w;
            w.x = dev::pack_act2(x.x, x.y, p.o16);
            w.y = dev::pack_act2(x.z, x.w, p.o16);
            *reinterpret_cast<uint2*>(p.o + ridx * D + c) = w;
          } else {
            *reinterpret_cast<float4*>(p.opart + ((long long)split * plane + ridx) * D + c) = x;
          }
        }
      }
    }
  }

teardown:
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::kTmemCols));
  }
}

}  // namespace

cudaError_t attn_tc_setup() {
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       TcCfg<64>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              TcCfg<128>::kSmem);
}

cudaError_t launch_attention_tc(const AttnParams& p, int d, cudaStream_t st) {
  const dim3 grid(p.row_tiles, p.nsplit, p.Hkv);
  if (d == 128) return launch_k(attn_tc_kernel<128>, grid, kThreads, TcCfg<128>::kSmem, st, p);
  return launch_k(attn_tc_kernel<64>, grid, kThreads, TcCfg<64>::kSmem, st, p);
}

}  // namespace kvr
