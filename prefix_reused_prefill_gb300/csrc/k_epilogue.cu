// Row-wise kernels around the projections: RoPE tables, the first RMSNorm,
// and the epilogues that add the k-split partial sums of a projection in a
// fixed order and then
//   * QKV:    rotate q and k (rotate-half RoPE at the row's absolute slot
//             position), round to bf16, write q and append k, v to the slot;
//   * resid:  add to the fp32 residual stream, then RMSNorm the new row for
//             the next projection (or write the bf16 output);
//   * swiglu: silu(gate) * up -> bf16;
//   * cast:   bf16 output of an attention-only layer.
// goinfer "What goinfer does": a conversation keeps one key and one value row
// per token and layer; a row's K/V land at its slot position so later turns
// reuse them.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = 0.f;
  const int nw = blockDim.x >> 5;
  for (int i = 0; i < nw; ++i) t += red[i];
  return t;
}

__device__ __forceinline__ float split_sum(const float* part, long long plane, int ksplit,
                                           long long idx) {
  float v = 0.f;
  for (int s = 0; s < ksplit; ++s) v += part[s * plane + idx];
  return v;
}

// cos/sin of pos * theta^(-2j/d), evaluated in double and rounded once.
__device__ __forceinline__ float2 rope_pair(const RowMap& rows, int i, int j, const RopeFreq& fr) {
  const double ang = (double)row_pos(rows, i) * fr.inv[j];
  double sn, cs;
  sincos(ang, &sn, &cs);
  return make_float2((float)cs, (float)sn);
}

__global__ void rope_table_kernel(RowMap rows, int d, RopeFreq fr, float2* table) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const int half = d / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows.m * half) return;
  table[idx] = rope_pair(rows, idx / half, idx % half, fr);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One CTA (256 threads) per row i: the row's RoPE pairs (threads j < d/2), h =
// float(hidden) and a = act(h * rsqrt(mean(h^2) + eps) * gain).  Each thread
// holds its 8-element vectors of the row in registers between the sum and the
// scaling (all of the row for H <= 4096; beyond that the rest is re-read).
__global__ void __launch_bounds__(256) embed_kernel(const __nv_bfloat16* hidden, int H, const __nv_bfloat16* gain,
                                                    float eps, float* h, __nv_bfloat16* a, bool a16, RowMap rows,
                                                    int half, RopeFreq fr, float2* table) {
  dev::pdl_trigger();
  __shared__ float red[32];
  constexpr int kV = 2;
  const int i = blockIdx.x;
  const long long row = i;
  const int H8 = H >> 3;
  // the norm gains are weights (no launch writes them): requested before the wait
  const uint4* g8 = reinterpret_cast<const uint4*>(gain);
  uint4 gv[kV];
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int k8 = threadIdx.x + u * 256;
    gv[u] = gain && k8 < H8 ? g8[k8] : make_uint4(0u, 0u, 0u, 0u);
  }
  dev::pdl_wait();
  if (table && (int)threadIdx.x < half) table[row * half + threadIdx.x] = rope_pair(rows, i, threadIdx.x, fr);
  const uint4* src = reinterpret_cast<const uint4*>(hidden + row * H);
  uint4* dst = reinterpret_cast<uint4*>(a + row * H);
  uint4 v[kV];
  float ss = 0.f;
  auto sq = [](const uint4& x) {
    float t = 0.f;
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) t += bf16_lo(w[q]) * bf16_lo(w[q]) + bf16_hi(w[q]) * bf16_hi(w[q]);
    return t;
  };
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int k8 = threadIdx.x + u * 256;
    v[u] = k8 < H8 ? src[k8] : make_uint4(0u, 0u, 0u, 0u);
    ss += sq(v[u]);
  }
  if (!gain) {   // attention-only layer: the input rows are the projection's input
    auto copy = [&](const uint4& x, int k8) {
      uint4 o;
      o.x = dev::pack_act2(bf16_lo(x.x), bf16_hi(x.x), a16);
      o.y = dev::pack_act2(bf16_lo(x.y), bf16_hi(x.y), a16);
      o.z = dev::pack_act2(bf16_lo(x.z), bf16_hi(x.z), a16);
      o.w = dev::pack_act2(bf16_lo(x.w), bf16_hi(x.w), a16);
      dst[k8] = o;
    };
#pragma unroll
    for (int u = 0; u < kV; ++u)
      if ((int)threadIdx.x + u * 256 < H8) copy(v[u], threadIdx.x + u * 256);
    for (int k8 = threadIdx.x + kV * 256; k8 < H8; k8 += 256) copy(src[k8], k8);
    return;
  }
  for (int k8 = threadIdx.x + kV * 256; k8 < H8; k8 += 256) ss += sq(src[k8]);
  const float rs = rsqrtf(block_sum(ss, red) / H + eps);
  float4* h4 = reinterpret_cast<float4*>(h + row * H);
  auto put = [&](const uint4& x, const uint4& g, int k8) {
    const float f[8] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y),
                        bf16_lo(x.z), bf16_hi(x.z), bf16_lo(x.w), bf16_hi(x.w)};
    const float gf[8] = {bf16_lo(g.x), bf16_hi(g.x), bf16_lo(g.y), bf16_hi(g.y),
                         bf16_lo(g.z), bf16_hi(g.z), bf16_lo(g.w), bf16_hi(g.w)};
    h4[2 * k8] = make_float4(f[0], f[1], f[2], f[3]);
    h4[2 * k8 + 1] = make_float4(f[4], f[5], f[6], f[7]);
    uint4 o;
    o.x = dev::pack_act2(f[0] * rs * gf[0], f[1] * rs * gf[1], a16);
    o.y = dev::pack_act2(f[2] * rs * gf[2], f[3] * rs * gf[3], a16);
    o.z = dev::pack_act2(f[4] * rs * gf[4], f[5] * rs * gf[5], a16);
    o.w = dev::pack_act2(f[6] * rs * gf[6], f[7] * rs * gf[7], a16);
    dst[k8] = o;
  };
#pragma unroll
  for (int u = 0; u < kV; ++u)
    if ((int)threadIdx.x + u * 256 < H8) put(v[u], gv[u], threadIdx.x + u * 256);
  for (int k8 = threadIdx.x + kV * 256; k8 < H8; k8 += 256) put(src[k8], g8[k8], k8);
}

// One CTA per row: a = bf16(h * rsqrt(mean(h^2) + eps) * gain), the RMSNorm
// of a row of the fp32 residual stream (float4 loads; the row stays in
// registers between the sum and the scaling for H <= 4096).
__global__ void __launch_bounds__(256) norm_kernel(const float* h, int H, const __nv_bfloat16* gain, float eps,
                                                   __nv_bfloat16* a) {
  dev::pdl_trigger();
  __shared__ float red[32];
  constexpr int kV = 4;   // float4 per thread held in registers
  const long long row = blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(h + row * H);
  const int H4 = H >> 2;
  // the gains are weights (no launch writes them): requested before the wait
  const uint2* g2 = reinterpret_cast<const uint2*>(gain);
  uint2 gw[kV];
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int k4 = threadIdx.x + u * 256;
    gw[u] = k4 < H4 ? g2[k4] : make_uint2(0u, 0u);
  }
  dev::pdl_wait();
  float4 v[kV];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int k4 = threadIdx.x + u * 256;
    v[u] = k4 < H4 ? src[k4] : make_float4(0.f, 0.f, 0.f, 0.f);
    ss += v[u].x * v[u].x + v[u].y * v[u].y + v[u].z * v[u].z + v[u].w * v[u].w;
  }
  for (int k4 = threadIdx.x + kV * 256; k4 < H4; k4 += 256) {
    const float4 x = src[k4];
    ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
  }
  const float rs = rsqrtf(block_sum(ss, red) / H + eps);
  auto put = [&](const float4& x, const uint2& g, int k4) {
    const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&g.x);
    const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&g.y);
    uint2 o;
    o.x = dev::pack_bf16x2(x.x * rs * __bfloat162float(g01.x), x.y * rs * __bfloat162float(g01.y));
    o.y = dev::pack_bf16x2(x.z * rs * __bfloat162float(g23.x), x.w * rs * __bfloat162float(g23.y));
    reinterpret_cast<uint2*>(a + row * H)[k4] = o;
  };
#pragma unroll
  for (int u = 0; u < kV; ++u) {
    const int k4 = threadIdx.x + u * 256;
    if (k4 < H4) put(v[u], gw[u], k4);
  }
  for (int k4 = threadIdx.x + kV * 256; k4 < H4; k4 += 256) put(src[k4], g2[k4], k4);
}

// One CTA per (tile of tokens, head): sum the split partials, rotate q/k
// (pair j, j + d/2), round to bf16; q rows go to the KV-head-major q buffer,
// K rows to the slot, and V through a shared-memory transpose to the slot's
// V^T rows so every global write is contiguous.  Thread = (token, 8-pair chunk).
template <int D>
__global__ void __launch_bounds__(256, 4) epi_qkv_kernel(const float* part, long long plane, int ksplit,
                                                      int ldo, int c0, int mb, RowMap rows, int Hq,
                                                      int Hkv, const float2* rope, __nv_bfloat16* q,
                                                      __nv_bfloat16* arena, long long k_off,
                                                      long long v_off, long long slot_stride, int cap) {
  dev::pdl_trigger();
  dev::pdl_wait();
  constexpr int kHalf = D / 2;
  constexpr int kChunks = kHalf / 8;          // threads per token
  constexpr int kTok = 256 / kChunks;         // tokens per CTA
  __shared__ __nv_bfloat16 vt[kTok][D + 8];
  const int hd = blockIdx.y;
  const int tl = threadIdx.x / kChunks, ch = threadIdx.x % kChunks;
  const int t = blockIdx.x * kTok + tl;
  const bool live = t < mb;
  const int i = c0 + t;
  const int j0 = 8 * ch;
  float x1[8], x2[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) x1[e] = x2[e] = 0.f;
  // (cos, sin) of pairs j0 .. j0+7, loaded alongside the split partials
  float4 cs[4];
  const bool rotate = live && hd < Hq + Hkv;
  if (rotate) {
    const float4* cs4 = reinterpret_cast<const float4*>(rope + (long long)i * kHalf + j0);
#pragma unroll
    for (int e = 0; e < 4; ++e) cs[e] = cs4[e];
  }
  if (live) {
    const float* src = part + (long long)t * ldo + (long long)hd * D + j0;
#pragma unroll 4
    for (int s = 0; s < ksplit; ++s) {
      const float4 a0 = *reinterpret_cast<const float4*>(src + s * plane);
      const float4 a1 = *reinterpret_cast<const float4*>(src + s * plane + 4);
      const float4 b0 = *reinterpret_cast<const float4*>(src + s * plane + kHalf);
      const float4 b1 = *reinterpret_cast<const float4*>(src + s * plane + kHalf + 4);
      x1[0] += a0.x; x1[1] += a0.y; x1[2] += a0.z; x1[3] += a0.w;
      x1[4] += a1.x; x1[5] += a1.y; x1[6] += a1.z; x1[7] += a1.w;
      x2[0] += b0.x; x2[1] += b0.y; x2[2] += b0.z; x2[3] += b0.w;
      x2[4] += b1.x; x2[5] += b1.y; x2[6] += b1.z; x2[7] += b1.w;
    }
  }
  if (hd < Hq + Hkv) {
    if (rotate) {
      float y1[8], y2[8];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const float4 c = cs[e / 2];   // (cos, sin) of pairs j0+e and j0+e+1
        y1[e] = x1[e] * c.x - x2[e] * c.y;
        y2[e] = x2[e] * c.x + x1[e] * c.y;
        y1[e + 1] = x1[e + 1] * c.z - x2[e + 1] * c.w;
        y2[e + 1] = x2[e + 1] * c.z + x1[e + 1] * c.w;
      }
      __nv_bfloat16* dst;
      if (hd < Hq) {
        const int G = Hq / Hkv;
        dst = q + q_row(rows, i, hd / G, hd % G, G, Hq) * D;
      } else {
        dst = arena + k_off + row_slot(rows, i) * slot_stride + ((long long)(hd - Hq) * cap + row_store(rows, i)) * D;
      }
      uint4 lo, hi;
      lo.x = dev::pack_bf16x2(y1[0], y1[1]); lo.y = dev::pack_bf16x2(y1[2], y1[3]);
      lo.z = dev::pack_bf16x2(y1[4], y1[5]); lo.w = dev::pack_bf16x2(y1[6], y1[7]);
      hi.x = dev::pack_bf16x2(y2[0], y2[1]); hi.y = dev::pack_bf16x2(y2[2], y2[3]);
      hi.z = dev::pack_bf16x2(y2[4], y2[5]); hi.w = dev::pack_bf16x2(y2[6], y2[7]);
      *reinterpret_cast<uint4*>(dst + j0) = lo;
      *reinterpret_cast<uint4*>(dst + kHalf + j0) = hi;
    }
  } else {
    // V: stage the tile, then write V^T rows [d][positions] of this head
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      vt[tl][j0 + e] = __float2bfloat16_rn(x1[e]);
      vt[tl][kHalf + j0 + e] = __float2bfloat16_rn(x2[e]);
    }
    __syncthreads();
    const int ntok = min(kTok, mb - (int)blockIdx.x * kTok);
    const int t0 = c0 + blockIdx.x * kTok;
    __nv_bfloat16* base = arena + v_off + (long long)(hd - Hq - Hkv) * D * cap;
    for (int idx = threadIdx.x; idx < D * kTok; idx += 256) {
      const int e = idx / kTok, tt = idx % kTok;
      if (tt < ntok)
        base[row_slot(rows, t0 + tt) * slot_stride + (long long)e * cap + row_store(rows, t0 + tt)] = vt[tt][e];
    }
  }
}

// One CTA per token row: h += sum of the split partials (fixed split order),
// then RMSNorm of the new row for the next projection, or the bf16 output.
// 512 threads x V float4; every split's loads of a thread are issued before
// any of them is added (the kernel is L2-latency-bound), and the row stays in
// registers between the two passes.
constexpr int kResidThreads = 512;
template <int V>  // float4 per thread (H <= 4 * 512 * V)
__global__ void __launch_bounds__(kResidThreads, V <= 2 ? 2 : 1) epi_resid_kernel(const float* part, long long plane, int ksplit,
                                                                  int ldo, int c0, int H, float* h,
                                                                  const __nv_bfloat16* gain, float eps,
                                                                  __nv_bfloat16* a_out, bool a16,
                                                                  __nv_bfloat16* final_out) {
  dev::pdl_trigger();
  __shared__ float red[32];
  const int t = blockIdx.x;
  const long long i = c0 + t;
  const int H4 = H >> 2;
  // the norm gains are weights (no launch writes them): requested before the wait
  uint2 gw[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int k4 = threadIdx.x + u * kResidThreads;
    gw[u] = a_out && k4 < H4 ? reinterpret_cast<const uint2*>(gain)[k4] : make_uint2(0u, 0u);
  }
  dev::pdl_wait();
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4* pp = reinterpret_cast<const float4*>(part + (long long)t * ldo);
  const long long pl4 = plane >> 2;
  // splits in flight at once: five (a 5-way k-split in one round) for up to
  // two float4 per thread, which keeps two CTAs on an SM (62 registers), so
  // one wave covers 304 rows
  constexpr int kB = V <= 2 ? 5 : kGemmMaxSplit / 2;
  float4 v[V];
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int k4 = threadIdx.x + u * kResidThreads;
    v[u] = k4 < H4 ? reinterpret_cast<const float4*>(h + i * H)[k4] : zero;
  }
  for (int s0 = 0; s0 < ksplit; s0 += kB) {
    float4 q[kB][V];
#pragma unroll
    for (int s = 0; s < kB; ++s)
#pragma unroll
      for (int u = 0; u < V; ++u) {
        const int k4 = threadIdx.x + u * kResidThreads;
        q[s][u] = (s0 + s < ksplit && k4 < H4) ? pp[(s0 + s) * pl4 + k4] : zero;
      }
    // h + p0 + p1 + ... in split order
#pragma unroll
    for (int s = 0; s < kB; ++s)
#pragma unroll
      for (int u = 0; u < V; ++u)
        if (s0 + s < ksplit) {
          v[u].x += q[s][u].x; v[u].y += q[s][u].y; v[u].z += q[s][u].z; v[u].w += q[s][u].w;
        }
  }
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int k4 = threadIdx.x + u * kResidThreads;
    if (k4 < H4) {
      const float4 acc = v[u];
      reinterpret_cast<float4*>(h + i * H)[k4] = acc;
      ss += acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
      if (final_out) {
        uint2 o;
        o.x = dev::pack_bf16x2(acc.x, acc.y);
        o.y = dev::pack_bf16x2(acc.z, acc.w);
        reinterpret_cast<uint2*>(final_out + i * H)[k4] = o;
      }
    }
  }
  if (a_out) {
    const float rs = rsqrtf(block_sum(ss, red) / H + eps);
#pragma unroll
    for (int u = 0; u < V; ++u) {
      const int k4 = threadIdx.x + u * kResidThreads;
      if (k4 < H4) {
        const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&gw[u].x);
        const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&gw[u].y);
        uint2 o;
        o.x = dev::pack_act2(v[u].x * rs * __bfloat162float(g01.x), v[u].y * rs * __bfloat162float(g01.y), a16);
        o.y = dev::pack_act2(v[u].z * rs * __bfloat162float(g23.x), v[u].w * rs * __bfloat162float(g23.y), a16);
        reinterpret_cast<uint2*>(a_out + i * H)[k4] = o;
      }
    }
  }
}

__global__ void epi_swiglu_kernel(const float* part, long long plane, int ksplit, int ldo, int c0,
                                  int mb, int F, __nv_bfloat16* z) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)mb * F) return;
  const int t = (int)(idx / F), n = (int)(idx % F);
  const float g = split_sum(part, plane, ksplit, (long long)t * ldo + n);
  const float u = split_sum(part, plane, ksplit, (long long)t * ldo + F + n);
  const float sg = g / (1.f + expf(-g));
  z[(long long)(c0 + t) * F + n] = __float2bfloat16_rn(sg * u);
}

__global__ void epi_cast_kernel(const float* part, long long plane, int ksplit, int ldo, int c0,
                                int mb, int N, __nv_bfloat16* out, bool f16) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)mb * N) return;
  const int t = (int)(idx / N), n = (int)(idx % N);
  dev::store_act(out + (long long)(c0 + t) * N + n, split_sum(part, plane, ksplit, (long long)t * ldo + n), f16);
}

inline unsigned blocks_for(long long n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

RopeFreq rope_freq(float theta, int d) {
  RopeFreq fr;
  for (int j = 0; j < 64; ++j) fr.inv[j] = j < d / 2 ? pow((double)theta, -2.0 * j / d) : 0.0;
  return fr;
}

cudaError_t launch_rope_table(const RowMap& rows, int d, const RopeFreq& fr, float2* table, cudaStream_t st) {
  const long long n = (long long)rows.m * (d / 2);
  return launch_k(rope_table_kernel, blocks_for(n, 256), 256, 0, st, rows, d, fr, table);
}

cudaError_t launch_embed(const __nv_bfloat16* hidden, int m, int H, const __nv_bfloat16* gain,
                         float eps, float* h, __nv_bfloat16* a, bool a16, const RowMap& rows, int d,
                         const RopeFreq& fr, float2* table, cudaStream_t st) {
  if (H % 8 || d / 2 > 64) return cudaErrorInvalidValue;
  return launch_k(embed_kernel, m, 256, 0, st, hidden, H, gain, eps, h, a, a16, rows, d / 2, fr, table);
}

cudaError_t launch_norm(const float* h, int m, int H, const __nv_bfloat16* gain, float eps,
                        __nv_bfloat16* a, cudaStream_t st) {
  if (H % 4) return cudaErrorInvalidValue;
  return launch_k(norm_kernel, m, 256, 0, st, h, H, gain, eps, a);
}

// One warp per token: the largest of the tiles' bests, lowest row on ties.
__global__ void __launch_bounds__(256) head_argmax_kernel(const float2* best, int tiles, int m, int32_t* out) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= m) return;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int k = lane; k < tiles; k += 32) {
    const float2 v = best[(long long)t * tiles + k];
    const int i = (int)v.y;
    if (v.x > bv || (v.x == bv && i < bi)) { bv = v.x; bi = i; }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  if (lane == 0) out[t] = bi;
}

cudaError_t launch_head_argmax(const float2* best, int tiles, int m, int32_t* out, cudaStream_t st) {
  return launch_k(head_argmax_kernel, (m + 7) / 8, 256, 0, st, best, tiles, m, out);
}

// One bounded wait on an mbarrier that nothing completes: it gives up after
// the wait limit and records the timeout in the status word.
__global__ void wait_probe_kernel(int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  dev::mbar_init(dev::smem_u32(&bar), 1);
  dev::fence_mbar_init();
  dev::mbar_wait(dev::smem_u32(&bar), 0, status);
}

cudaError_t launch_wait_probe(int* status, cudaStream_t st) {
  wait_probe_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_epi_qkv(const float* part, long long plane, int ksplit, int ldo, int c0, int mb,
                           const RowMap& rows, int Hq, int Hkv, int d, const float2* rope,
                           __nv_bfloat16* q, __nv_bfloat16* arena, long long k_off,
                           long long v_off, long long slot_stride, int cap, cudaStream_t st) {
  const int heads = Hq + 2 * Hkv;
  if (d == 128) {
    const dim3 grid((mb + 15) / 16, heads);
    return launch_k(epi_qkv_kernel<128>, grid, 256, 0, st, part, plane, ksplit, ldo, c0, mb, rows, Hq,
                    Hkv, rope, q, arena, k_off, v_off, slot_stride, cap);
  } else if (d == 64) {
    const dim3 grid((mb + 31) / 32, heads);
    return launch_k(epi_qkv_kernel<64>, grid, 256, 0, st, part, plane, ksplit, ldo, c0, mb, rows, Hq,
                    Hkv, rope, q, arena, k_off, v_off, slot_stride, cap);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_epi_resid(const float* part, long long plane, int ksplit, int ldo, int c0,
                             int mb, int H, float* h, const __nv_bfloat16* gain, float eps,
                             __nv_bfloat16* a_out, bool a16, __nv_bfloat16* final_out, cudaStream_t st) {
  if (ksplit > kGemmMaxSplit) return cudaErrorInvalidValue;
  const int v = (H / 4 + kResidThreads - 1) / kResidThreads;
  if (v <= 1)
    return launch_k(epi_resid_kernel<1>, mb, kResidThreads, 0, st, part, plane, ksplit, ldo, c0, H, h, gain,
                    eps, a_out, a16, final_out);
  if (v <= 2)
    return launch_k(epi_resid_kernel<2>, mb, kResidThreads, 0, st, part, plane, ksplit, ldo, c0, H, h, gain,
                    eps, a_out, a16, final_out);
  if (v <= 4)
    return launch_k(epi_resid_kernel<4>, mb, kResidThreads, 0, st, part, plane, ksplit, ldo, c0, H, h, gain,
                    eps, a_out, a16, final_out);
  return cudaErrorInvalidValue;
}

cudaError_t launch_epi_swiglu(const float* part, long long plane, int ksplit, int ldo, int c0,
                              int mb, int F, __nv_bfloat16* z, cudaStream_t st) {
  return launch_k(epi_swiglu_kernel, blocks_for((long long)mb * F, 256), 256, 0, st, part, plane,
                  ksplit, ldo, c0, mb, F, z);
}

cudaError_t launch_epi_cast(const float* part, long long plane, int ksplit, int ldo, int c0,
                            int mb, int N, __nv_bfloat16* out, bool f16, cudaStream_t st) {
  return launch_k(epi_cast_kernel, blocks_for((long long)mb * N, 256), 256, 0, st, part, plane,
                  ksplit, ldo, c0, mb, N, out, f16);
}

}  // namespace kvr
