// Large-m projections on the 5th-generation tensor cores: Y = X W^T with int4
// group-32 weights, X bf16 [tokens][K], fp32 accumulation in tensor memory.
//
// thinkspread, "The economics of speculative decoding" (cost model): weights
// are read once and shared by all m rows.  At the m = 254 rows of goinfer's
// turn-9 replay the projections are a real dense contraction (3.3 TFLOP per
// 28-layer step), so they run as tcgen05.mma instead of a GEMV.
//
// One CTA = 128 weight rows x up to 256 tokens (one tcgen05.mma M=128, N<=256
// tile, K = 16 per instruction), over a range of the K dimension (split-K for
// narrow projections).  Warp roles:
//   warp 0     TMA producer: int4 tile + fp16 scales (256 inputs per stage,
//              128B-swizzled, 2 stages) and activation tiles (64 inputs x N
//              tokens, 128B-swizzled K-major, 3 stages);
//   warp 1     allocates the TMEM accumulator; one thread issues tcgen05.mma
//              and tcgen05.commit (which frees the smem stages it read);
//   warps 2-17 converters: int4 codes -> bf16 weights (code * scale, exact for
//              scales with at most 8 significant bits) written as 128B-swizzled
//              K-major A tiles.  Four groups of four warps: group g converts
//              atom g (inputs 64g..64g+63) of every 256-input chunk into its
//              own A stage, so four atoms are in flight at once and the latency
//              of one conversion (dequant, stores, proxy fence) is overlapped;
//              thread = (tile row, one of the atom's two 32-input groups).
//              Then the epilogue, the four groups taking 32-token chunks in
//              turn: tcgen05.ld of the accumulator, and either fp32 partial
//              sums (reduced row-wise by the epilogue kernels) or, for the
//              gate|up projection, the fused SwiGLU product silu(gate) * up.
// Every wait is bounded; on a timeout the CTA records it in the status word,
// drains its own copies and frees its TMEM before returning.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kConvGroups = 4;                  // one per 64-input atom of a 256-input chunk
constexpr int kConvWarps = 4 * kConvGroups;      // 4 warps (128 rows x 2 groups) per atom
constexpr int kThreads = 64 + 32 * kConvWarps;   // + producer warp + MMA warp
constexpr int kRawStages = 3;
constexpr int kPrefetch = 2;   // int4 chunks prefetched into L2 ahead of their TMA load
constexpr int kAStages = 4;
constexpr int kXStages = 3;
constexpr int kRawWBytes = 128 * 128;   // 128 rows x 256 inputs of int4
constexpr int kRawSBytes = 128 * 16;    // 128 rows x 8 fp16 scales
constexpr int kRawBytes = kRawWBytes + kRawSBytes;
constexpr int kABytes = 128 * 128;      // 128 rows x 64 inputs bf16
constexpr int kXMaxBytes = 256 * 128;   // 256 tokens x 64 inputs bf16
constexpr int kTmemCols = 256;
constexpr int kSmem = kRawStages * kRawBytes + kAStages * kABytes + kXStages * kXMaxBytes + 1024;

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
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

// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major.
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

// 8 codes of one 32-bit word -> 4 bf16x2 code values (field i low, field i+4 high)
__device__ __forceinline__ void codes_of_word(uint32_t w, __nv_bfloat162 out[4]) {
  const uint32_t magic = 0x43004300u;
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(magic));
    out[i] = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&v), bias);
  }
}

__global__ void __launch_bounds__(kThreads, 1) gemm_int4_tc_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t raw_full[kRawStages], raw_empty[kRawStages];
  __shared__ __align__(8) uint64_t a_full[kAStages], a_empty[kAStages];
  __shared__ __align__(8) uint64_t x_full[kXStages], x_empty[kXStages];
  __shared__ __align__(8) uint64_t acc_full;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint32_t raw_base = base;
  const uint32_t a_base = raw_base + kRawStages * kRawBytes;
  const uint32_t x_base = a_base + kAStages * kABytes;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // tile -> segment / rows; split -> range of 256-input chunks
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
  const int natoms = 4 * nkc;
  const uint32_t xbytes = (uint32_t)p.xrows * 128u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRawStages; ++i) {
      dev::mbar_init(dev::smem_u32(&raw_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&raw_empty[i]), kConvWarps);
    }
    for (int i = 0; i < kAStages; ++i) {
      dev::mbar_init(dev::smem_u32(&a_full[i]), kConvWarps / kConvGroups);
      dev::mbar_init(dev::smem_u32(&a_empty[i]), 1);
    }
    for (int i = 0; i < kXStages; ++i) {
      dev::mbar_init(dev::smem_u32(&x_full[i]), 1);
      dev::mbar_init(dev::smem_u32(&x_empty[i]), 1);
    }
    dev::mbar_init(dev::smem_u32(&acc_full), 1);
    *abort_v = 0;
    dev::fence_mbar_init();
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

  if (warp == 0) {
    // ---------------------------------------------------------------- producers
    // lane 0 streams int4 tiles + scales, lane 1 streams activation tiles; the
    // two rings are independent so neither stream waits behind the other.
    if (lane == 0) {
      dev::prefetch_tmap(&seg.tw);
      dev::prefetch_tmap(&seg.ts);
      const uint64_t pol = dev::policy_evict_first();
      auto prefetch_chunk = [&](int i) {
        const int kc = kc0 + i;
        if (p.swiglu) {
          dev::tma_prefetch_2d(&p.seg[0].tw, kc * 128, row0);
          dev::tma_prefetch_2d(&p.seg[1].tw, kc * 128, row0);
        } else {
          dev::tma_prefetch_2d(&seg.tw, kc * 128, row0);
        }
      };
      for (int i = 0; i < kPrefetch && i < nkc; ++i) prefetch_chunk(i);
      int raw_issued = 0;
      for (int i = 0; i < nkc; ++i) {
        if (i + kPrefetch < nkc) prefetch_chunk(i + kPrefetch);
        const int rs = i % kRawStages;
        if (i >= kRawStages &&
            (!dev::mbar_wait(dev::smem_u32(&raw_empty[rs]), ((i / kRawStages) - 1) & 1, p.status) ||
             *abort_v)) {
          *abort_v = 1;
          break;
        }
        const uint32_t rb = raw_base + rs * kRawBytes;
        const uint32_t fb = dev::smem_u32(&raw_full[rs]);
        dev::mbar_arrive_expect_tx(fb, kRawBytes);
        const int kc = kc0 + i;
        if (p.swiglu) {
          const GemmSeg& up = p.seg[1];
          dev::tma_load_2d_hint(rb, &p.seg[0].tw, kc * 128, row0, fb, pol);
          dev::tma_load_2d_hint(rb + kRawWBytes / 2, &up.tw, kc * 128, row0, fb, pol);
          dev::tma_load_2d_hint(rb + kRawWBytes, &p.seg[0].ts, kc * 8, row0, fb, pol);
          dev::tma_load_2d_hint(rb + kRawWBytes + kRawSBytes / 2, &up.ts, kc * 8, row0, fb, pol);
        } else {
          dev::tma_load_2d_hint(rb, &seg.tw, kc * 128, row0, fb, pol);
          dev::tma_load_2d_hint(rb + kRawWBytes, &seg.ts, kc * 8, row0, fb, pol);
        }
        ++raw_issued;
      }
      for (int st = 0; st < kRawStages && st < raw_issued; ++st) {
        const int last = ((raw_issued - 1 - st) / kRawStages) * kRawStages + st;
        dev::mbar_wait(dev::smem_u32(&raw_full[st]), (uint32_t)(last / kRawStages) & 1, nullptr);
      }
    } else if (lane == 1) {
      dev::prefetch_tmap(&p.tx);
      int x_issued = 0;
      for (int j = 0; j < natoms; ++j) {
        const int xs = j % kXStages;
        if (j >= kXStages &&
            (!dev::mbar_wait(dev::smem_u32(&x_empty[xs]), ((j / kXStages) - 1) & 1, p.status) ||
             *abort_v)) {
          *abort_v = 1;
          break;
        }
        const uint32_t xb = dev::smem_u32(&x_full[xs]);
        dev::mbar_arrive_expect_tx(xb, xbytes);
        dev::tma_load_2d(x_base + xs * kXMaxBytes, &p.tx, (kc0 + (j >> 2)) * 256 + 64 * (j & 3), p.t0, xb);
        ++x_issued;
      }
      for (int st = 0; st < kXStages && st < x_issued; ++st) {
        const int last = ((x_issued - 1 - st) / kXStages) * kXStages + st;
        dev::mbar_wait(dev::smem_u32(&x_full[st]), (uint32_t)(last / kXStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, p.n_tok);
      bool ok = true;
      for (int j = 0; j < natoms; ++j) {
        const int as = j % kAStages, xs = j % kXStages;
        if (!dev::mbar_wait(dev::smem_u32(&a_full[as]), (j / kAStages) & 1, p.status) ||
            !dev::mbar_wait(dev::smem_u32(&x_full[xs]), (j / kXStages) & 1, p.status) || *abort_v) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t ad = sw128_desc(a_base + as * kABytes);
        const uint64_t bd = sw128_desc(x_base + xs * kXMaxBytes);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem, ad + 2 * kk, bd + 2 * kk, idesc, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(dev::smem_u32(&a_empty[as]));
        mma_commit(dev::smem_u32(&x_empty[xs]));
      }
      if (!ok) *abort_v = 1;
      mma_commit(dev::smem_u32(&acc_full));
    }
  } else {
    // ---------------------------------------------------------------- converters
    const int cw = warp - 2;                 // 0..15
    const int grp = cw >> 2;                 // atom within each 256-input chunk = A stage
    const int cv = ((cw & 3) << 5) | lane;   // 0..127 within the group
    const int t = cv & 127;                  // tile row; the thread converts both 32-input groups
    bool ok = true;
    for (int i = 0; i < nkc && ok; ++i) {
      const int rs = i % kRawStages;
      ok = dev::mbar_wait(dev::smem_u32(&raw_full[rs]), (i / kRawStages) & 1, p.status) && !*abort_v;
      if (ok && i >= 1)
        ok = dev::mbar_wait(dev::smem_u32(&a_empty[grp]), (i - 1) & 1, p.status) && !*abort_v;
      if (!ok) break;
      const uint32_t rb = raw_base + rs * kRawBytes;
      uint32_t scw;  // fp16 scales of groups 2*grp (low half) and 2*grp+1 (high half)
      asm volatile("ld.shared.b32 %0, [%1];" : "=r"(scw) : "r"(rb + kRawWBytes + t * 16 + grp * 4));
      const uint4 w0 = dev::lds128(rb + dev::swz128(t, 2 * grp));
      const uint4 w1 = dev::lds128(rb + dev::swz128(t, 2 * grp + 1));
      const uint32_t ab = a_base + grp * kABytes + t * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 wv = h ? w1 : w0;
        const uint16_t sbits = (uint16_t)(h ? (scw >> 16) : (scw & 0xFFFFu));
        const float sf = __half2float(__ushort_as_half(sbits));
        const __nv_bfloat162 s2 = __floats2bfloat162_rn(sf, sf);
        __nv_bfloat162 c0[4], c1[4], c2[4], c3[4];
        codes_of_word(wv.x, c0);
        codes_of_word(wv.y, c1);
        codes_of_word(wv.z, c2);
        codes_of_word(wv.w, c3);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          __nv_bfloat162 v0 = __hmul2(c0[jj], s2), v1 = __hmul2(c1[jj], s2);
          __nv_bfloat162 v2 = __hmul2(c2[jj], s2), v3 = __hmul2(c3[jj], s2);
          const uint32_t chunk = (uint32_t)(4 * h + jj);
          const uint32_t addr = ab + ((chunk ^ (uint32_t)(t & 7)) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                       "r"(*reinterpret_cast<uint32_t*>(&v0)), "r"(*reinterpret_cast<uint32_t*>(&v1)),
                       "r"(*reinterpret_cast<uint32_t*>(&v2)), "r"(*reinterpret_cast<uint32_t*>(&v3))
                       : "memory");
        }
      }
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        dev::mbar_arrive(dev::smem_u32(&a_full[grp]));
        dev::mbar_arrive(dev::smem_u32(&raw_empty[rs]));
      }
    }
    if (!ok) *abort_v = 1;

    // ---------------------------------------------------------------- epilogue
    const bool have = __all_sync(0xffffffffu, dev::mbar_wait(dev::smem_u32(&acc_full), 0, p.status) && !*abort_v);
    tc_fence_after();
    if (have) {
      const int q = warp & 3;              // TMEM lane quarter this warp may read
      const int set = (warp - 2) >> 2;     // 0..3: the converter group of this warp
      const int trow = 32 * q + lane;      // tile row of this thread
      const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
      if (!p.swiglu) {
        const int row = row0 + trow;
        float* out = p.part + (long long)split * p.plane + seg.col0 + row;
        for (int c0 = 32 * set; c0 < p.n_tok; c0 += 32 * kConvGroups) {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          if (row < seg.N) {
#pragma unroll
            for (int k = 0; k < 32; ++k)
              if (c0 + k < p.m) out[(long long)(c0 + k) * p.ldo] = __uint_as_float(r[k]);
          }
        }
      } else {
        // rows 0..63 are gate, 64..127 the matching up rows: exchange through smem
        float* xch = reinterpret_cast<float*>(smem_raw + (a_base - dev::smem_u32(smem_raw))) + set * 64 * 33;
        const int n = row0 + (trow & 63);
        for (int c0 = 32 * set; c0 < p.n_tok; c0 += 32 * kConvGroups) {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          if (q >= 2) {
#pragma unroll
            for (int k = 0; k < 32; ++k) xch[(trow - 64) * 33 + k] = __uint_as_float(r[k]);
          }
          named_sync(1 + set, 128);
          if (q < 2 && n < seg.N) {
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              if (c0 + k < p.m) {
                const float g = __uint_as_float(r[k]);
                const float u = xch[trow * 33 + k];
                const float sg = g / (1.f + expf(-g));
                p.z[(long long)(p.t0 + c0 + k) * p.F + n] = __float2bfloat16_rn(sg * u);
              }
            }
          }
          named_sync(1 + set, 128);
        }
      }
    }
  }

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
  return cudaFuncSetAttribute(gemm_int4_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
}

cudaError_t launch_gemm_int4_tc(const GemmParams& p, int total_tiles, cudaStream_t st) {
  const dim3 grid(total_tiles, p.ksplit);
  gemm_int4_tc_kernel<<<grid, kThreads, kSmem, st>>>(p);
  return cudaGetLastError();
}

}  // namespace kvr
