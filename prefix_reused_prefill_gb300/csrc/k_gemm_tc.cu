// Large-m projections on the 5th-generation tensor cores: Y = X W^T with int4
// group-32 weights, fp32 accumulation in tensor memory.  Both operands are
// fp16: X [tokens][K] holds the activations' bf16 values (the model's rounding
// point) in fp16, which represents them exactly, and each dequantised weight
// code * scale is rounded once to fp16 (relative error at most 2^-12; the
// product of a 4-bit code and an 11-bit fp16 scale can need 14 bits).  The
// exact variant (the QKV projection, whose q and k feed a softmax that can
// amplify their errors) carries each weight as two fp16 terms, hi = fp16(w)
// and lo = fp16(w - hi) (the remainder has at most 4 significant bits), and
// issues both MMAs: twice the tensor work for exact weights.
//
// thinkspread, "The economics of speculative decoding" (cost model): each
// weight streams once for all m rows.  At the m = 254 rows of goinfer's
// turn-9 replay the projections are a real dense contraction (3.3 TFLOP per
// 28-layer step), so they run as tcgen05.mma instead of a GEMV.
//
// One CTA = 128 weight rows x up to 256 tokens (one tcgen05.mma M=128, N<=256
// tile, K = 16 per instruction), over a range of the K dimension (split-K for
// narrow projections).  The pipeline stage is 128 inputs, so the MMA thread
// issues 8 MMAs (1024 tensor cycles at N=256) per pair of barrier waits: a
// single issuing thread pays ~100-250 cycles per wait and ~60 per MMA, so
// smaller stages leave the tensor pipe idle.  The dequantised weights (the A
// operand) live in tensor memory, which keeps shared memory for a 3-deep
// activation ring.  Warp roles:
//   warp 0     lane 0 streams int4 tiles (128 inputs x 128 rows, 64B-swizzled,
//              4 stages, prefetched into L2 two stages ahead; it is thread 0,
//              which fills the ring as soon as it has initialised the
//              barriers, before the CTA's barrier), lane 1 streams
//              activation tiles (128 inputs x N tokens as two 128B-swizzled
//              K-major atoms, 3 stages); the two rings are independent;
//   warp 1     allocates the TMEM accumulator; one thread issues tcgen05.mma
//              and tcgen05.commit (which frees the smem stages it read);
//   warps 2-17 converters: int4 codes -> fp16 weights (code * scale rounded
//              once; the fp16 scales are read from global memory) stored
//              straight into a TMEM A stage with one
//              tcgen05.st per thread (thread = TMEM lane / tile row, one
//              64-input half of the stage).  Two groups of eight warps take
//              alternate stages of a 4-deep A ring in TMEM.
//              Then the epilogue, four sets of four warps taking 32-token
//              chunks in turn: tcgen05.ld of the accumulator, and either fp32
//              partial sums (reduced row-wise by the epilogue kernels) or, for
//              the gate|up projection, the fused SwiGLU product silu(gate)*up.
// Every wait is bounded; on a timeout the CTA records it in the status word,
// drains its own copies and frees its TMEM before returning.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kConvGroups = 2;                  // one per A stage
constexpr int kGroupWarps = 8;                   // 128 rows x two 64-input halves
constexpr int kConvWarps = kConvGroups * kGroupWarps;
constexpr int kThreads = 64 + 32 * kConvWarps;   // + producer warp + MMA warp
// The two converter groups take alternate stages, so the int4 ring has an even
// number of slots: each slot is then always consumed by the same group, one use
// after the other (a group never waits on a slot whose previous use belongs to
// the other group, which the mbarrier phase parity could not tell apart).
constexpr int kRawStages = 4;
constexpr int kStages = 3;                       // activation stages (shared memory)
constexpr int kAStages = 4;                      // A stages (tensor memory); 2 hi|lo stages when exact
constexpr int kPrefetch = 2;                     // int4 stages prefetched into L2 ahead
constexpr int kRawBytes = 128 * 64;              // 128 rows x 128 inputs of int4
constexpr int kXAtom = 256 * 128;                // one 64-input atom of up to 256 tokens
constexpr int kXBytes = 2 * kXAtom;
constexpr int kTmemCols = 512;                   // accumulator 256 + 4 A stages x 64 columns
constexpr uint32_t kACol = 256;                  // first A stage column; stage s at kACol + 64 s (128 s exact)
constexpr int kSmem = kRawStages * kRawBytes + kStages * kXBytes + 1024;

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// K-major operand in the 128-byte swizzle layout: 8-row atoms of 128-byte rows,
// atoms 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}

// kind::f16 instruction descriptor: D fp32, A and B fp16 (format fields 0),
// both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
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

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t r[32]) {
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
}

__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 8 codes of one 32-bit word -> 4 fp16x2 code values (field i low, field i+4
// high): the field OR'd into the mantissa of fp16 1024.0 is 1024 + field
// (the fp16 step is 1 there), and 1024 + field - 1032 = code, exactly.
__device__ __forceinline__ void codes_of_word(uint32_t w, __half2 out[4]) {
  const uint32_t magic = 0x64006400u;
  const __half2 bias = __floats2half2_rn(1032.0f, 1032.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(magic));
    out[i] = __hsub2(*reinterpret_cast<__half2*>(&v), bias);
  }
}

// K-quant: 8 unsigned 4-bit codes of one word -> 4 fp16x2 weights
// fp16(d*sc*q - dmin*mn) (pair i: fields i and i+4, as codes_of_word).  The
// codes become exact fp32 values 128 + q (the bf16 pattern 128 + q shifted
// into the high half), so w = (128 + q)*a + c with a = d*sc and
// c = -(128*a + dmin*mn), one fp32 FMA per weight on the full-rate pipe (c
// carries at most one fp32 rounding, far below the fp16 rounding that follows).
__device__ __forceinline__ void q4k_weights_of_word(uint32_t w, float a, float c, uint32_t out[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43004300u));
    const float ql = __uint_as_float(v << 16), qh = __uint_as_float(v & 0xFFFF0000u);
    __half2 hv = __floats2half2_rn(fmaf(ql, a, c), fmaf(qh, a, c));
    out[i] = *reinterpret_cast<uint32_t*>(&hv);
  }
}

// Exact variant: 8 4-bit fields of one word -> 4 pairs of weights w = (128 + f)*a + c
// formed in fp32 (exact for int4: a = scale, c = -136*scale gives code*scale)
// and split into fp16 hi = fp16(w) and lo = fp16(w - hi) (pair i: fields i, i+4).
__device__ __forceinline__ void hilo_weights_of_word(uint32_t w, float a, float c, uint32_t hi[4], uint32_t lo[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43004300u));
    const float wl = fmaf(__uint_as_float(v << 16), a, c), wh = fmaf(__uint_as_float(v & 0xFFFF0000u), a, c);
    __half2 h = __floats2half2_rn(wl, wh);
    const float2 f = __half22float2(h);
    __half2 l = __floats2half2_rn(wl - f.x, wh - f.y);
    hi[i] = *reinterpret_cast<uint32_t*>(&h);
    lo[i] = *reinterpret_cast<uint32_t*>(&l);
  }
}

__device__ __forceinline__ uint32_t q4k_field6(const uint4& r, int f) {
  const int p = 6 * f, word = p >> 5, off = p & 31;
  const uint32_t lo = word == 0 ? r.y : (word == 1 ? r.z : r.w);
  const uint32_t hi = word == 0 ? r.z : r.w;
  return (off > 26 && word < 2 ? __funnelshift_r(lo, hi, off) : lo >> off) & 63u;
}

template <bool kExact>
__global__ void __launch_bounds__(kThreads, 1) gemm_int4_tc_kernel(const __grid_constant__ GemmParams p) {
  constexpr int kAS = kExact ? 2 : kAStages;            // A stages in flight
  constexpr uint32_t kAW = kExact ? 128u : 64u;         // TMEM columns per A stage (hi, then lo)
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  __shared__ __align__(8) uint64_t a_full[kAStages], a_empty[kAStages];
  __shared__ __align__(8) uint64_t x_full[kStages], x_empty[kStages];
  __shared__ __align__(8) uint64_t acc_full;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  __shared__ int epi_bad;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t raw_base = base;
  const uint32_t x_base = raw_base + kRawStages * kRawBytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile -> segment / rows; split -> range of 128-input stages
  const int tile = blockIdx.x;
  int s = 0;
  while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile0) ++s;
  const GemmSeg& seg = p.seg[s];
  const int rows_per_tile = p.swiglu ? 64 : 128;
  const int row0 = (tile - seg.tile0) * rows_per_tile;
  const int split = blockIdx.y;
  const int kc0 = (int)((long long)split * p.kchunks / p.ksplit);
  const int kc1 = (int)((long long)(split + 1) * p.kchunks / p.ksplit);
  const int nkc = kc1 - kc0;
  const uint32_t xbytes = 2u * (uint32_t)p.xrows * 128u;

  // the int4 stream of stage i (thread 0: the weight producer)
  auto prefetch_stage = [&](int i) {
    const int x = (kc0 + i) * 64;
    if (p.swiglu) {
      dev::tma_prefetch_2d(&p.seg[0].tw, x, row0);
      dev::tma_prefetch_2d(&p.seg[1].tw, x, row0);
    } else {
      dev::tma_prefetch_2d(&seg.tw, x, row0);
    }
  };
  auto load_stage = [&](int i, uint64_t pol) {
    const int rs = i % kRawStages;
    const uint32_t rb = raw_base + rs * kRawBytes;
    const uint32_t fb = dev::smem_u32(&raw_full[rs]);
    dev::mbar_arrive_expect_tx(fb, kRawBytes);
    const int x = (kc0 + i) * 64;
    if (p.swiglu) {
      dev::tma_load_2d_hint(rb, &p.seg[0].tw, x, row0, fb, pol);
      dev::tma_load_2d_hint(rb + kRawBytes / 2, &p.seg[1].tw, x, row0, fb, pol);
    } else {
      dev::tma_load_2d_hint(rb, &seg.tw, x, row0, fb, pol);
    }
  };
  // int4 stages the weight producer issues before the CTA's barrier
  const int early = nkc < kRawStages ? nkc : kRawStages;

  dev::pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      dev::mbar_init(dev::smem_u32(&raw_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&raw_empty[i]), kGroupWarps);
    }
    for (int i = 0; i < kAS; ++i) {
      dev::mbar_init(dev::smem_u32(&a_full[i]), kGroupWarps);
      dev::mbar_init(dev::smem_u32(&a_empty[i]), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&x_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&x_empty[i]), 1);
    }
    dev::mbar_init(dev::smem_u32(&acc_full), 1);
    // a wait has given up earlier in the call: the CTA issues no copy and
    // runs no role (one decision for the whole CTA, taken after the
    // allocation's barrier: a barrier of its own before the allocation cost
    // the projection kernels ~10 % of their time)
    *abort_v = dev::status_set(p.status) ? 1 : 0;
    epi_bad = 0;
    dev::fence_mbar_init();
    // Thread 0 is also the weight producer: it fills the int4 ring now (its
    // barriers are initialised and fenced), while warp 1 allocates TMEM, so the
    // first stage's HBM latency overlaps the CTA's set-up.  Weights depend on
    // no earlier launch.
    if (!*abort_v) {
      dev::prefetch_tmap(&p.seg[0].tw);
      if (p.swiglu) dev::prefetch_tmap(&p.seg[1].tw);
      else dev::prefetch_tmap(&seg.tw);
      const uint64_t pol = dev::policy_evict_first();
      for (int i = 0; i < early; ++i) load_stage(i, pol);
      for (int i = early; i < early + kPrefetch && i < nkc; ++i) prefetch_stage(i);
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dev::smem_u32(&tmem_slot)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (*abort_v) goto teardown;
  // Only the activation stream (warp 0, lane 1) and, before it writes, the
  // epilogue depend on the previous launch: the int4 stream, the converters
  // (weights and scales) and the MMA issuer (fed by the two streams) run
  // ahead, so the A stages are full when the activations arrive.
  if (warp == 0 && lane == 1) dev::pdl_wait();

  if (warp == 0) {
    // ---------------------------------------------------------------- producers
    if (lane == 0) {
      // stages 0 .. early-1 went out before the CTA's barrier (thread 0)
      const uint64_t pol = dev::policy_evict_first();
      int issued = early;
      for (int i = early; i < nkc; ++i) {
        if (i + kPrefetch < nkc) prefetch_stage(i + kPrefetch);
        const int rs = i % kRawStages;
        if (i >= kRawStages &&
            (!dev::mbar_wait(dev::smem_u32(&raw_empty[rs]), ((i / kRawStages) - 1) & 1, p.status) ||
             *abort_v)) {
          *abort_v = 1;
          break;
        }
        load_stage(i, pol);
        ++issued;
      }
      const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
      for (int st = 0; st < kRawStages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / kRawStages) * kRawStages + st;
        dev::mbar_wait_until(dev::smem_u32(&raw_full[st]), (uint32_t)(last / kRawStages) & 1, deadline);
      }
    } else if (lane == 1) {
      dev::prefetch_tmap(&p.tx);
      int issued = 0;
      for (int i = 0; i < nkc; ++i) {
        const int st = i % kStages;
        if (i >= kStages &&
            (!dev::mbar_wait(dev::smem_u32(&x_empty[st]), ((i / kStages) - 1) & 1, p.status) || *abort_v)) {
          *abort_v = 1;
          break;
        }
        const uint32_t xb = dev::smem_u32(&x_full[st]);
        dev::mbar_arrive_expect_tx(xb, xbytes);
        const uint32_t dst = x_base + st * kXBytes;
        dev::tma_load_2d(dst, &p.tx, (kc0 + i) * 128, p.t0, xb);
        dev::tma_load_2d(dst + kXAtom, &p.tx, (kc0 + i) * 128 + 64, p.t0, xb);
        ++issued;
      }
      const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / kStages) * kStages + st;
        dev::mbar_wait_until(dev::smem_u32(&x_full[st]), (uint32_t)(last / kStages) & 1, deadline);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16(128, p.n_tok);
      bool ok = true;
      for (int i = 0; i < nkc; ++i) {
        const int xs = i % kStages, as = i % kAS;
        if (!dev::mbar_wait(dev::smem_u32(&a_full[as]), (i / kAS) & 1, p.status) ||
            !dev::mbar_wait(dev::smem_u32(&x_full[xs]), (i / kStages) & 1, p.status) || *abort_v) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t ta = tmem + kACol + kAW * (uint32_t)as;
#pragma unroll
        for (int atom = 0; atom < 2; ++atom) {
          const uint64_t bd = sw128_desc(x_base + xs * kXBytes + atom * kXAtom);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            mma_f16_ta(tmem, ta + 32u * atom + 8u * kk, bd + 2 * kk, idesc,
                       (i > 0 || atom > 0 || kk > 0) ? 1u : 0u);
            if (kExact) mma_f16_ta(tmem, ta + 64u + 32u * atom + 8u * kk, bd + 2 * kk, idesc, 1u);
          }
        }
        mma_commit(dev::smem_u32(&a_empty[as]));
        mma_commit(dev::smem_u32(&x_empty[xs]));
      }
      if (!ok) *abort_v = 1;
      mma_commit(dev::smem_u32(&acc_full));
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int cw = warp - 2;                      // 0..15
    const int grp = cw / kGroupWarps;             // stages grp, grp+2, ... (A stage i % 4)
    const int q = warp & 3;                       // TMEM lane quarter this warp may write
    const int hq = ((cw % kGroupWarps) >> 2) & 1; // 64-input half of the stage
    const int t = 32 * q + lane;                  // tile row = TMEM lane
    // fp16 scales of this row: gate / up rows for the SwiGLU tile
    const GemmSeg& sseg = (p.swiglu && t >= 64) ? p.seg[1] : seg;
    const int srow = p.swiglu ? row0 + (t & 63) : row0 + t;
    const bool srow_ok = srow < sseg.N;
    const int G = p.K / 32;
    const uint32_t* sptr = reinterpret_cast<const uint32_t*>(sseg.scales + (long long)(srow_ok ? srow : 0) * G);
    // K-quant: the row's 16-byte superblock records (same row stride, K/32 halves)
    const uint4* rptr = reinterpret_cast<const uint4*>(sptr);
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    bool ok = true;
    for (int i = grp; i < nkc; i += kConvGroups) {
      const int rs = i % kRawStages, as = i % kAS;
      // scales of groups 4*(kc0+i) + 2*hq and +1 (one aligned 32-bit load), or
      // the K-quant record of superblock (kc0+i)/2 (sub-blocks 4*((kc0+i)&1) + 2*hq, +1)
      uint32_t scw = 0u;
      uint4 rec = make_uint4(0u, 0u, 0u, 0u);
      if (p.fmt == kFmtQ4K) {
        if (srow_ok) rec = __ldg(rptr + (kc0 + i) / 2);
      } else {
        scw = srow_ok ? __ldg(sptr + 2 * (kc0 + i) + hq) : 0u;
      }
      ok = dev::mbar_wait(dev::smem_u32(&raw_full[rs]), (i / kRawStages) & 1, p.status) && !*abort_v;
      if (ok && i >= kAS)
        ok = dev::mbar_wait(dev::smem_u32(&a_empty[as]), ((i / kAS) - 1) & 1, p.status) && !*abort_v;
      if (!__all_sync(0xffffffffu, ok)) {
        ok = false;
        break;
      }
      const uint32_t rb = raw_base + rs * kRawBytes + t * 64;
      const uint32_t sw = (uint32_t)((t >> 1) & 3);  // 64-byte swizzle of this row
      const uint4 w0 = dev::lds128(rb + (((uint32_t)(2 * hq) ^ sw) << 4));
      const uint4 w1 = dev::lds128(rb + (((uint32_t)(2 * hq + 1) ^ sw) << 4));
      const uint32_t abase = tmem + tlane + kACol + kAW * (uint32_t)as + 32u * (uint32_t)hq;
      if constexpr (kExact) {
        // hi and lo of the 64 weights of this row (k order, two per column)
        uint32_t hi[32], lo[32];
        const float d = __half2float(__ushort_as_half((unsigned short)(rec.x & 0xFFFFu)));
        const float dmin = __half2float(__ushort_as_half((unsigned short)(rec.x >> 16)));
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 wv = h ? w1 : w0;
          float a, c;
          if (p.fmt == kFmtQ4K) {
            const int j = 4 * ((kc0 + i) & 1) + 2 * hq + h;
            a = d * (float)q4k_field6(rec, j);
            c = -fmaf(128.f, a, dmin * (float)q4k_field6(rec, 8 + j));
          } else {
            a = __half2float(__ushort_as_half((uint16_t)(h ? (scw >> 16) : (scw & 0xFFFFu))));
            c = -136.f * a;
          }
          uint32_t h4[4][4], l4[4][4];
          hilo_weights_of_word(wv.x, a, c, h4[0], l4[0]);
          hilo_weights_of_word(wv.y, a, c, h4[1], l4[1]);
          hilo_weights_of_word(wv.z, a, c, h4[2], l4[2]);
          hilo_weights_of_word(wv.w, a, c, h4[3], l4[3]);
#pragma unroll
          for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              hi[16 * h + 4 * jj + wi] = h4[wi][jj];
              lo[16 * h + 4 * jj + wi] = l4[wi][jj];
            }
        }
        tmem_st32(abase, hi);
        tmem_st32(abase + 64u, lo);
      } else {
        uint32_t outv[32];   // 64 fp16 weights of this row, k order, two per column
        if (p.fmt == kFmtQ4K) {
          const float d = __half2float(__ushort_as_half((unsigned short)(rec.x & 0xFFFFu)));
          const float dmin = __half2float(__ushort_as_half((unsigned short)(rec.x >> 16)));
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 wv = h ? w1 : w0;
            const int j = 4 * ((kc0 + i) & 1) + 2 * hq + h;   // sub-block of the superblock
            const float a = d * (float)q4k_field6(rec, j);
            const float c = -fmaf(128.f, a, dmin * (float)q4k_field6(rec, 8 + j));
            uint32_t c0[4], c1[4], c2[4], c3[4];
            q4k_weights_of_word(wv.x, a, c, c0);
            q4k_weights_of_word(wv.y, a, c, c1);
            q4k_weights_of_word(wv.z, a, c, c2);
            q4k_weights_of_word(wv.w, a, c, c3);
  #pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
              outv[16 * h + 4 * jj + 0] = c0[jj];
              outv[16 * h + 4 * jj + 1] = c1[jj];
              outv[16 * h + 4 * jj + 2] = c2[jj];
              outv[16 * h + 4 * jj + 3] = c3[jj];
            }
          }
        } else {
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint4 wv = h ? w1 : w0;
          const uint16_t sbits = (uint16_t)(h ? (scw >> 16) : (scw & 0xFFFFu));
          const __half2 s2 = __half2half2(__ushort_as_half(sbits));
          __half2 c0[4], c1[4], c2[4], c3[4];
          codes_of_word(wv.x, c0);
          codes_of_word(wv.y, c1);
          codes_of_word(wv.z, c2);
          codes_of_word(wv.w, c3);
  #pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            // inputs 8*jj .. 8*jj+7 of this 32-input group: words 0..3 give pairs (2w, 2w+1)
            // code * scale: the exact product rounded once to fp16
            __half2 v0 = __hmul2(c0[jj], s2), v1 = __hmul2(c1[jj], s2);
            __half2 v2 = __hmul2(c2[jj], s2), v3 = __hmul2(c3[jj], s2);
            outv[16 * h + 4 * jj + 0] = *reinterpret_cast<uint32_t*>(&v0);
            outv[16 * h + 4 * jj + 1] = *reinterpret_cast<uint32_t*>(&v1);
            outv[16 * h + 4 * jj + 2] = *reinterpret_cast<uint32_t*>(&v2);
            outv[16 * h + 4 * jj + 3] = *reinterpret_cast<uint32_t*>(&v3);
          }
        }
        }
        tmem_st32(abase, outv);
      }
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        dev::mbar_arrive(dev::smem_u32(&a_full[as]));
        dev::mbar_arrive(dev::smem_u32(&raw_empty[rs]));
      }
    }
    if (!ok) *abort_v = 1;

    // ---------------------------------------------------------------- epilogue
    // one decision for all sixteen epilogue warps (the SwiGLU sets' barriers
    // need all of their warps)
    const bool have_w = __all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&acc_full), 0, p.status) && !*abort_v);
    if (!have_w && lane == 0) epi_bad = 1;
    tc_fence_after();
    dev::pdl_wait();   // the outputs below may still be read by the previous launch
    named_sync(5, 32 * kConvWarps);
    const bool have = epi_bad == 0;
    if (have) {
      const int set = cw >> 2;             // 0..3
      const int trow = 32 * q + lane;      // tile row of this thread
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
      if (!p.swiglu) {
        const int row = row0 + trow;
        float* out = p.part + (long long)split * p.plane + seg.col0 + row;
        for (int c0 = 32 * set; c0 < p.n_tok; c0 += 128) {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          if (row < seg.N) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (c0 + k < p.m) out[(long long)(c0 + k) * p.ldo] = __uint_as_float(r[k]);
          }
        }
      } else {
        // rows 0..63 are gate, 64..127 the matching up rows: each warp stages
        // its 32 rows x 32 tokens in shared memory, then the set's 128 threads
        // form z = silu(g) * u for 64 rows x 32 tokens (thread = row, token parity)
        float* xch = reinterpret_cast<float*>(smem_raw + (x_base - dev::smem_u32(smem_raw))) + set * 128 * 33;
        const int tid = 32 * q + lane;       // 0..127 within the set
        const int r = tid & 63, kp = tid >> 6;
        const int n = row0 + r;
        for (int c0 = 32 * set; c0 < p.n_tok; c0 += 128) {
          uint32_t v[32];
          tmem_ld32(taddr + c0, v);
#pragma unroll
          for (int k = 0; k < 32; ++k) xch[trow * 33 + k] = __uint_as_float(v[k]);
          named_sync(1 + set, 128);
          if (n < seg.N) {
#pragma unroll
            for (int k = kp; k < 32; k += 2) {
              if (c0 + k < p.m) {
                const float g = xch[r * 33 + k];
                const float u = xch[(64 + r) * 33 + k];
                const float sg = __fdividef(g, 1.f + __expf(-g));
                dev::store_act(p.z + (long long)(p.t0 + c0 + k) * p.F + n, sg * u, p.z16 != 0);
              }
            }
          }
          named_sync(1 + set, 128);
        }
      }
    }
  }

teardown:
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
}

}  // namespace

int gemm_tc_smem() { return kSmem; }

cudaError_t gemm_tc_setup() {
  cudaError_t e = cudaFuncSetAttribute(gemm_int4_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_int4_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  return e;
}

cudaError_t launch_gemm_int4_tc(const GemmParams& p, int total_tiles, cudaStream_t st) {
  const dim3 grid(total_tiles, p.ksplit);
  return p.exact ? launch_k(gemm_int4_tc_kernel<true>, grid, kThreads, kSmem, st, p)
                 : launch_k(gemm_int4_tc_kernel<false>, grid, kThreads, kSmem, st, p);
}

}  // namespace kvr
