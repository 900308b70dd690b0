// m-row batched GEMV: Y[t][n] = sum_k X[t][k] * W[n][k] for up to 32 token rows,
// each weight byte read from HBM once for all rows.
//
// thinkspread, "The economics of speculative decoding" (cost model): the m
// verify rows run as a batched GEMV whose weights are read once and shared by
// the rows, so an extra row costs far less than a full weight read.
//
// int4 group-32 path (the hot one).  A CTA owns 128 weight rows and a range of
// 256-input k-steps.  One producer warp streams, per k-step, a 128 x 128-byte
// int4 tile (128B-swizzled), its 128 x 8 fp16 scales and the 8*NT x 256 bf16
// activation tile through TMA into a multi-stage shared-memory ring guarded by
// mbarriers.  Eight consumer warps each own 16 weight rows:
//   * one 32-bit shared load per row gives a thread the eight 4-bit codes it
//     needs for the two m16n8k16 fragments of one 32-input group (the byte
//     layout of include/kvr.h is chosen for this);
//   * codes become exact bf16 integers (code+8 OR'd into the mantissa of 128.0,
//     minus 136);
//   * the unscaled group product sum_k code*x runs on the tensor cores with an
//     fp32 accumulator, and the fp16 group scale is applied afterwards in fp32:
//     acc += scale * group_sum.  The weight is therefore exactly code*scale,
//     never rounded to bf16.
// Plain CUDA-core FMAs would need 32*m FMAs per 16 weight bytes, more than the
// SM issues at HBM rate once m > 2; the tensor cores keep the kernel HBM-bound.
// Partial sums for each k-split go to a fp32 buffer; a row-wise epilogue
// kernel adds the splits in a fixed order and applies the fused epilogue.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kConsumerWarps = kGemvRows / 16;   // 8
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kWTileBytes = kGemvRows * 128;       // 16 KB
constexpr int kSTileBytes = kGemvRows * 16;        // 2 KB

template <int NT>
struct GemvCfg {
  static constexpr int kXRows = 8 * NT;
  static constexpr int kXBoxBytes = kXRows * 128;             // one 64-input box
  static constexpr int kXTileBytes = 4 * kXBoxBytes;          // 256 inputs
  static constexpr int kStageBytes = kWTileBytes + kXTileBytes + kSTileBytes;
  static constexpr int kStages = 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024;  // + alignment slack
};

// 8 int4 codes of one 32-bit word -> 4 bf16x2 registers holding code values.
// Register i holds fields i (low half) and i+4 (high half).
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t r[4]) {
  const uint32_t magic = 0x43004300u;  // bf16 128.0 in both halves
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    const uint32_t s = w >> (4 * i);
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(s), "r"(0x000F000Fu), "r"(magic));
    __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
    h = __hsub2(h, bias);
    r[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) gemv_int4_kernel(const __grid_constant__ GemvParams p) {
  using C = GemvCfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // which segment / row tile / k range
  const int tile = blockIdx.x;
  int s = 0;
  while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile0) ++s;
  const GemvSeg& seg = p.seg[s];
  const int row0 = (tile - seg.tile0) * kGemvRows;
  const int split = blockIdx.y;
  const int ks0 = (int)((long long)split * p.ksteps / p.ksplit);
  const int ks1 = (int)((long long)(split + 1) * p.ksteps / p.ksplit);
  const int nk = ks1 - ks0;

  dev::pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&full_bar[i]), 1);
      dev::mbar_init(dev::smem_u32(&empty_bar[i]), kConsumerWarps);
    }
    *abort_v = 0;
    dev::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      dev::prefetch_tmap(&seg.tw);
      dev::prefetch_tmap(&seg.ts);
      dev::prefetch_tmap(&p.tx);
      const uint64_t pol = dev::policy_evict_first();
      // Weights do not depend on earlier launches: fill the ring's weight and
      // scale tiles and pull the rest of this CTA's weights toward L2 before
      // waiting for the previous launch; the activations follow the wait.
      const int pre = nk < C::kStages ? nk : C::kStages;
      for (int it = 0; it < pre; ++it) {
        const uint32_t sb = base + it * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&full_bar[it]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        dev::tma_load_2d_hint(sb, &seg.tw, (ks0 + it) * 128, row0, fb, pol);
        dev::tma_load_2d_hint(sb + kWTileBytes + C::kXTileBytes, &seg.ts, (ks0 + it) * 8, row0, fb, pol);
      }
      for (int it = pre; it < nk; ++it) {
        dev::tma_prefetch_2d(&seg.tw, (ks0 + it) * 128, row0);
        dev::tma_prefetch_2d(&seg.ts, (ks0 + it) * 8, row0);
      }
      dev::pdl_wait();
      for (int it = 0; it < pre; ++it) {
        const uint32_t sb = base + it * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&full_bar[it]);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dev::tma_load_2d(sb + kWTileBytes + j * C::kXBoxBytes, &p.tx, (ks0 + it) * kGemvKStep + 64 * j,
                           p.c0, fb);
      }
      int issued = pre;
      for (int it = pre; it < nk; ++it) {
        const int st = it % C::kStages;
        const uint32_t use = (uint32_t)(it / C::kStages);
        if (!dev::mbar_wait(dev::smem_u32(&empty_bar[st]), (use - 1) & 1, p.status) || *abort_v) {
          *abort_v = 1;
          break;
        }
        const uint32_t sb = base + st * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&full_bar[st]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        const int ks = ks0 + it;
        dev::tma_load_2d_hint(sb, &seg.tw, ks * 128, row0, fb, pol);
        dev::tma_load_2d_hint(sb + kWTileBytes + C::kXTileBytes, &seg.ts, ks * 8, row0, fb, pol);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          dev::tma_load_2d(sb + kWTileBytes + j * C::kXBoxBytes, &p.tx, ks * kGemvKStep + 64 * j,
                           p.c0, fb);
        ++issued;
      }
      // never leave the CTA with copies in flight: wait (bounded) for the last
      // use of every stage that was filled
      for (int st = 0; st < C::kStages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / C::kStages) * C::kStages + st;
        dev::mbar_wait(dev::smem_u32(&full_bar[st]), (uint32_t)(last / C::kStages) & 1, nullptr);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  dev::pdl_wait();                  // the partial sums are written below
  const int r = lane >> 2;          // fragment row 0..7
  const int c = lane & 3;           // fragment column pair
  const int rho0 = warp * 16 + r;   // tile rows of this thread: rho0 and rho0+8
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;

  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  for (int it = 0; it < nk; ++it) {
    const int st = it % C::kStages;
    const uint32_t use = (uint32_t)(it / C::kStages);
    if (!dev::mbar_wait(dev::smem_u32(&full_bar[st]), use & 1, p.status) || *abort_v) {
      *abort_v = 1;
      break;
    }
    const uint32_t wt = base + st * C::kStageBytes;
    const uint32_t xt = wt + kWTileBytes;
    const uint32_t stile = xt + C::kXTileBytes;
    const uint4 sc0 = dev::lds128(stile + rho0 * 16);
    const uint4 sc1 = dev::lds128(stile + (rho0 + 8) * 16);
    const __half* s0h = reinterpret_cast<const __half*>(&sc0);
    const __half* s1h = reinterpret_cast<const __half*>(&sc1);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t w0 = dev::lds32(wt + dev::swz128(rho0, g) + 4 * c);
      const uint32_t w1 = dev::lds32(wt + dev::swz128(rho0 + 8, g) + 4 * c);
      uint32_t q0[4], q1[4];
      dequant_word(w0, q0);
      dequant_word(w1, q1);
      const uint32_t a_lo[4] = {q0[0], q1[0], q0[1], q1[1]};  // inputs 0..15 of the group
      const uint32_t a_hi[4] = {q0[2], q1[2], q0[3], q1[3]};  // inputs 16..31
      const float sr0 = __half2float(s0h[g]);
      const float sr1 = __half2float(s1h[g]);
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        // B fragments: tokens t*8 .. t*8+7, inputs 32g + 8q .. +7 for q = 0..3
        const int n = t * 8 + (lane & 7);
        const int q = lane >> 3;
        const int box = g >> 1;
        const int chunk = 4 * (g & 1) + q;
        uint32_t b0, b1, b2, b3;
        dev::ldmatrix_x4(xt + box * C::kXBoxBytes + dev::swz128(n, chunk), b0, b1, b2, b3);
        float tmp[4];
        dev::mma_bf16_16816(tmp, a_lo, b0, b1, zero4);
        dev::mma_bf16_16816(tmp, a_hi, b2, b3, tmp);
        acc[t][0] = fmaf(sr0, tmp[0], acc[t][0]);
        acc[t][1] = fmaf(sr0, tmp[1], acc[t][1]);
        acc[t][2] = fmaf(sr1, tmp[2], acc[t][2]);
        acc[t][3] = fmaf(sr1, tmp[3], acc[t][3]);
      }
    }
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[st]));
  }
  if (*abort_v) return;

  // write this split's partial sums: part[split][token][col0 + row]
  float* out = p.part + (long long)split * p.plane;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = t * 8 + 2 * c + (e & 1);
      const int row = row0 + rho0 + (e >> 1) * 8;
      if (tok < p.mb && row < seg.N) out[(long long)tok * p.ldo + seg.col0 + row] = acc[t][e];
    }
  }
}

// bf16 weights (the tiny attention-only shape and small bf16 stacks): one warp
// per output column, 16-byte loads along K, every token of the pass per warp.
__global__ void __launch_bounds__(256) gemv_bf16_kernel(const __grid_constant__ GemvParams p,
                                                        int total_cols) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp >= total_cols) return;
  int s = 0;
  while (s + 1 < p.nseg && warp >= p.seg[s + 1].col0) ++s;
  const GemvSeg& seg = p.seg[s];
  const int n = warp - seg.col0;
  const __nv_bfloat16* wrow = seg.wbf + (long long)n * p.K;
  float acc[kGemvMaxCols];
#pragma unroll
  for (int t = 0; t < kGemvMaxCols; ++t) acc[t] = 0.f;
  for (int k = lane * 8; k < p.K; k += 256) {
    const uint4 wv = *reinterpret_cast<const uint4*>(wrow + k);
    const __nv_bfloat16* wb = reinterpret_cast<const __nv_bfloat16*>(&wv);
    float wf[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) wf[j] = __bfloat162float(wb[j]);
#pragma unroll
    for (int t = 0; t < kGemvMaxCols; ++t) {
      if (t < p.mb) {
        const uint4 xv =
            *reinterpret_cast<const uint4*>(p.x + (long long)(p.c0 + t) * p.K + k);
        const __nv_bfloat16* xb = reinterpret_cast<const __nv_bfloat16*>(&xv);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[t] = fmaf(wf[j], __bfloat162float(xb[j]), acc[t]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kGemvMaxCols; ++t) {
    float v = acc[t];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && t < p.mb) p.part[(long long)t * p.ldo + warp] = v;
  }
}

}  // namespace

int gemv_int4_smem(int nt) {
  switch (nt) {
    case 1: return GemvCfg<1>::kSmem;
    case 2: return GemvCfg<2>::kSmem;
    default: return GemvCfg<4>::kSmem;
  }
}

cudaError_t gemv_setup() {
  cudaError_t e;
  e = cudaFuncSetAttribute(gemv_int4_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemvCfg<1>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(gemv_int4_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GemvCfg<2>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(gemv_int4_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              GemvCfg<4>::kSmem);
}

cudaError_t launch_gemv_int4(const GemvParams& p, int total_tiles, int nt, cudaStream_t st) {
  const dim3 grid(total_tiles, p.ksplit);
  switch (nt) {
    case 1: return launch_k(gemv_int4_kernel<1>, grid, kThreads, GemvCfg<1>::kSmem, st, p);
    case 2: return launch_k(gemv_int4_kernel<2>, grid, kThreads, GemvCfg<2>::kSmem, st, p);
    default: return launch_k(gemv_int4_kernel<4>, grid, kThreads, GemvCfg<4>::kSmem, st, p);
  }
}

cudaError_t launch_gemv_bf16(const GemvParams& p, int total_cols, cudaStream_t st) {
  const int blocks = (total_cols * 32 + 255) / 256;
  return launch_k(gemv_bf16_kernel, blocks, 256, 0, st, p, total_cols);
}

}  // namespace kvr
