// Causal grouped-query attention for many new rows on the 5th-generation
// tensor cores: S = Q K^T and P V as tcgen05.mma with accumulators in TMEM.
//
// goinfer, "Turn nine in under half a second" ("What goinfer does"): the 254
// new rows of turn 9 attend to the 1668 cached rows plus themselves; with
// all G query heads of a KV head packed as rows (row = token*G + head in the
// group), one KV head's rows form a real dense contraction.
//
// One CTA = (128-row tile of one KV head, key split).  Warp roles:
//   warp 0     TMA: the Q tile once (128 rows x d, 128B-swizzled K-major), then
//              per 64-key block a K tile ([64 keys][d]) and a V^T tile
//              ([d][64 keys]; V is stored transposed in the slot), 3 stages;
//   warp 1     allocates TMEM; one thread issues S_j = Q K_j^T (M=128, N=64)
//              into a double-buffered S accumulator and O += P_j V_j (M=128,
//              N=d) into one O accumulator that stays in TMEM for the whole
//              key range, software-pipelined so S_{j+1} is computed while the
//              softmax works on block j;
//   warps 2-5  one thread per row: tcgen05.ld of S_j, causal mask, online
//              softmax in fp32 (log2 units) and P_j written to shared memory as
//              a 128B-swizzled K-major bf16 tile.  The running-max correction of
//              O is lazy: P_j is taken relative to a per-row reference max, and
//              only when a block's max exceeds the reference by more than 8
//              (P would exceed 2^8) does the warp rescale its rows of O in TMEM
//              (tcgen05.ld / tcgen05.st) and move the reference.  At the end
//              O / l is written (or, with several key splits, the unnormalised
//              partials merged by attn_combine).
// Every wait is bounded; a timed-out CTA records it, drains its copies and
// frees its TMEM.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kKeys = 64;
constexpr int kThreads = 192;

template <int D>
struct TcCfg {
  static constexpr int kQBytes = 128 * D * 2;
  static constexpr int kKBytes = kKeys * D * 2;   // D/64 atoms of [64 keys][64 elems]
  static constexpr int kVBytes = D * kKeys * 2;   // one atom of [D rows][64 keys]
  static constexpr int kStageBytes = kKBytes + kVBytes;
  static constexpr int kStages = 3;
  static constexpr int kPBytes = 128 * kKeys * 2;
  static constexpr int kSmem = kQBytes + kStages * kStageBytes + kPBytes + 1024;
  // TMEM columns: S buffers at 0 and 64, the O accumulator at 128
  static __device__ __forceinline__ uint32_t scol(int b) { return (uint32_t)(64 * b); }
  static constexpr uint32_t kOCol = 128;
  static constexpr int kTmemCols = 256;
};

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
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
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
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
  __shared__ __align__(8) uint64_t kv_full[C::kStages], kv_empty[C::kStages];
  __shared__ __align__(8) uint64_t s_full[2], s_empty[2], p_full, pv_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t q_base = base;
  const uint32_t kv_base = q_base + C::kQBytes;
  const uint32_t p_base = kv_base + C::kStages * C::kStageBytes;
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
    for (int i = 0; i < C::kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&kv_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&kv_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      dev::mbar_init(dev::smem_u32(&s_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&s_empty[i]), 4);
    }
    dev::mbar_init(dev::smem_u32(&p_full), 4);
    dev::mbar_init(dev::smem_u32(&pv_done), 1);
    *abort_v = 0;
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
  // q and this call's K/V come from the previous launch; only the producer's
  // loads of cached-prefix K/V may run ahead of it.
  if (warp != 0 || lane != 0) dev::pdl_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0 && nblk == 0) dev::pdl_wait();
    if (lane == 0 && nblk > 0) {
      dev::prefetch_tmap(&p.tq);
      dev::prefetch_tmap(&p.tkv);
      dev::prefetch_tmap(&p.tvt);
      int pre = 0;
      while (pre < nblk && pre < C::kStages && (b0 + pre + 1) * kKeys <= p.rows.P) {
        const uint32_t sb = kv_base + pre * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&kv_full[pre]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        const int key0 = (b0 + pre) * kKeys;
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          dev::tma_load_2d(sb + a * (kKeys * 128), &p.tkv, 64 * a, p.kbase + kv * p.cap + key0, fb);
        dev::tma_load_2d(sb + C::kKBytes, &p.tvt, key0, p.vtbase + kv * D, fb);
        ++pre;
      }
      dev::pdl_wait();
      const uint32_t qb = dev::smem_u32(&q_full);
      dev::mbar_arrive_expect_tx(qb, C::kQBytes);
      const int qrow = kv * R + row_lo;
#pragma unroll
      for (int a = 0; a < D / 64; ++a) dev::tma_load_2d(q_base + a * 16384, &p.tq, 64 * a, qrow, qb);
      int issued = pre;
      for (int j = pre; j < nblk; ++j) {
        const int st = j % C::kStages;
        if (j >= C::kStages &&
            (!dev::mbar_wait(dev::smem_u32(&kv_empty[st]), ((j / C::kStages) - 1) & 1, p.status) ||
             *abort_v)) {
          *abort_v = 1;
          break;
        }
        const uint32_t sb = kv_base + st * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&kv_full[st]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        const int key0 = (b0 + j) * kKeys;
#pragma unroll
        for (int a = 0; a < D / 64; ++a)
          dev::tma_load_2d(sb + a * (kKeys * 128), &p.tkv, 64 * a, p.kbase + kv * p.cap + key0, fb);
        dev::tma_load_2d(sb + C::kKBytes, &p.tvt, key0, p.vtbase + kv * D, fb);
        ++issued;
      }
      dev::mbar_wait(qb, 0, nullptr);
      for (int st = 0; st < C::kStages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / C::kStages) * C::kStages + st;
        dev::mbar_wait(dev::smem_u32(&kv_full[st]), (uint32_t)(last / C::kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nblk > 0) {
      const uint32_t id_qk = idesc_bf16(128, kKeys);
      const uint32_t id_pv = idesc_bf16(128, D);
      bool ok = dev::mbar_wait(dev::smem_u32(&q_full), 0, p.status);
      auto pv = [&](int b) -> bool {
        const int st = b % C::kStages;
        if (!dev::mbar_wait(dev::smem_u32(&p_full), b & 1, p.status) || *abort_v) return false;
        tc_fence_after();
        const uint64_t pd = sw128_desc(p_base);
        const uint64_t vd = sw128_desc(kv_base + st * C::kStageBytes + C::kKBytes);
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          mma_f16(tmem + C::kOCol, pd + 2 * kk, vd + 2 * kk, id_pv, (b > 0 || kk > 0) ? 1u : 0u);
        mma_commit(dev::smem_u32(&pv_done));
        mma_commit(dev::smem_u32(&kv_empty[st]));
        return true;
      };
      for (int j = 0; j < nblk && ok; ++j) {
        const int st = j % C::kStages, sb = j & 1;
        if (!dev::mbar_wait(dev::smem_u32(&kv_full[st]), (j / C::kStages) & 1, p.status) ||
            (j >= 2 && !dev::mbar_wait(dev::smem_u32(&s_empty[sb]), ((j - 2) >> 1) & 1, p.status)) ||
            *abort_v) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t kd = sw128_desc(kv_base + st * C::kStageBytes);
        const uint64_t qd = sw128_desc(q_base);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_f16(tmem + C::scol(sb), qd + (kk >> 2) * (16384 >> 4) + 2 * (kk & 3),
                  kd + (kk >> 2) * ((kKeys * 128) >> 4) + 2 * (kk & 3), id_qk, kk > 0 ? 1u : 0u);
        mma_commit(dev::smem_u32(&s_full[sb]));
        if (j >= 1 && !pv(j - 1)) ok = false;
      }
      if (ok) ok = pv(nblk - 1);
      if (!ok) *abort_v = 1;
    }
  } else {
    // ---------------------------------------------------------------- softmax
    const int q4 = warp & 3;
    const int r = 32 * q4 + lane;
    const uint32_t tlane = (uint32_t)(32 * q4) << 16;
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
    bool ok = true;
    for (int j = 0; j < nblk && ok; ++j) {
      const int sb = j & 1;
      ok = dev::mbar_wait(dev::smem_u32(&s_full[sb]), (j >> 1) & 1, p.status) && !*abort_v;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[kKeys];
      tmem_ld32_nowait(tmem + tlane + C::scol(sb), sr);
      tmem_ld32_nowait(tmem + tlane + C::scol(sb) + 32, sr + 32);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_u32(&s_empty[sb]));
      const int key0 = (b0 + j) * kKeys;
      // visible keys of this row within the block: [0, P) and [lo, hi]
      const int pe = min(max(P0 - key0, 0), kKeys);            // keys k < pe are in [0, P)
      const int la = min(max(lo - key0, 0), kKeys);            // own range k in [la, hb)
      const int hb = tok >= 0 ? min(max(hi - key0 + 1, 0), kKeys) : 0;
      float s[kKeys];
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kKeys; ++k) {
        const bool vis = tok >= 0 && (k < pe || (k >= la && k < hb));
        s[k] = vis ? __uint_as_float(sr[k]) * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, s[k]);
      }
      // lazy reference max: move it (and rescale O) only when P would exceed 2^8
      const bool move = mx > m_ref + kLazyMax;
      const float m_new = move ? mx : m_ref;
      const float factor = (move && m_ref != -INFINITY) ? exp2f(m_ref - m_new) : 1.f;
      const float muse = m_new == -INFINITY ? 0.f : m_new;
      uint32_t pk[kKeys / 2];
      float sum = 0.f;
#pragma unroll
      for (int k = 0; k < kKeys; k += 2) {
        const float e0 = exp2f(s[k] - muse), e1 = exp2f(s[k + 1] - muse);
        sum += e0 + e1;
        pk[k / 2] = dev::pack_bf16x2(e0, e1);
      }
      // P V of block j-1 must be done: it reads the P buffer and accumulates into O
      if (j >= 1) {
        ok = dev::mbar_wait(dev::smem_u32(&pv_done), (j - 1) & 1, p.status) && !*abort_v;
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, factor != 1.f)) {
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t v[32];
            tmem_ld32_nowait(tmem + tlane + C::kOCol + c0, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * factor);
            tmem_st32(tmem + tlane + C::kOCol + c0, v);
          }
          tmem_wait_st();
        }
      }
      l = l * factor + sum;
      m_ref = m_new;
      const uint32_t prow = p_base + r * 128;
#pragma unroll
      for (int ch = 0; ch < 8; ++ch) {
        const uint32_t addr = prow + (((uint32_t)ch ^ (uint32_t)(r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * ch]),
                     "r"(pk[4 * ch + 1]), "r"(pk[4 * ch + 2]), "r"(pk[4 * ch + 3])
                     : "memory");
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_u32(&p_full));
    }
    if (ok && nblk > 0) {
      ok = dev::mbar_wait(dev::smem_u32(&pv_done), (nblk - 1) & 1, p.status) && !*abort_v;
      ok = __all_sync(0xffffffffu, ok);
    }
    if (!ok) *abort_v = 1;
    if (ok) {
      tc_fence_after();
      const long long rowidx = (long long)tok * p.Hq + head;
      const long long plane = (long long)p.rows.m * p.Hq;
      const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        if (nblk > 0) {
          tmem_ld32(tmem + tlane + C::kOCol + c0, v);
        } else {
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = 0.f;
        }
        if (tok >= 0) {
          if (p.nsplit == 1) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + rowidx * D + c0);
#pragma unroll
            for (int c8 = 0; c8 < 4; ++c8) {
              uint4 w;
              w.x = dev::pack_bf16x2(v[8 * c8] * inv, v[8 * c8 + 1] * inv);
              w.y = dev::pack_bf16x2(v[8 * c8 + 2] * inv, v[8 * c8 + 3] * inv);
              w.z = dev::pack_bf16x2(v[8 * c8 + 4] * inv, v[8 * c8 + 5] * inv);
              w.w = dev::pack_bf16x2(v[8 * c8 + 6] * inv, v[8 * c8 + 7] * inv);
              dst[c8] = w;
            }
          } else {
            float4* dst = reinterpret_cast<float4*>(p.opart + ((long long)split * plane + rowidx) * D + c0);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4)
              dst[c4] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
          }
        }
      }
      if (tok >= 0 && p.nsplit > 1) p.ml[split * plane + rowidx] = make_float2(m_ref, l);
    }
  }

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
