// Row-wise kernels around the projections: RoPE tables, the first RMSNorm,
// and the epilogues that add the k-split partial sums of a projection in a
// fixed order and then
//   * QKV:    rotate q and k (rotate-half RoPE at the row's absolute slot
//             position), round to bf16, write q and append k, v to the slot;
//   * resid:  add to the fp32 residual stream, then RMSNorm the new row for
//             the next projection (or write the bf16 output);
//   * swiglu: silu(gate) * up -> bf16;
//   * cast:   bf16 output of an attention-only layer.
// goinfer "What goinfer does": the KV cache is two vectors per token per
// layer; a row's K/V land at its slot position so later turns reuse them.
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
__global__ void rope_table_kernel(RowMap rows, int d, double theta, float2* table) {
  const int half = d / 2;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows.m * half) return;
  const int i = idx / half, j = idx % half;
  const int b = row_branch(rows, i);
  const double pos = (double)(rows.P + i - rows.off[b]);
  const double ang = pos * pow(theta, -2.0 * j / d);
  double sn, cs;
  sincos(ang, &sn, &cs);
  table[idx] = make_float2((float)cs, (float)sn);
}

__global__ void embed_kernel(const __nv_bfloat16* hidden, int H, const __nv_bfloat16* gain,
                             float eps, float* h, __nv_bfloat16* a) {
  __shared__ float red[32];
  const long long row = blockIdx.x;
  float ss = 0.f;
  for (int k = threadIdx.x; k < H; k += blockDim.x) {
    const float v = __bfloat162float(hidden[row * H + k]);
    h[row * H + k] = v;
    ss += v * v;
  }
  const float rs = rsqrtf(block_sum(ss, red) / H + eps);
  for (int k = threadIdx.x; k < H; k += blockDim.x)
    a[row * H + k] = __float2bfloat16_rn(h[row * H + k] * rs * __bfloat162float(gain[k]));
}

__global__ void epi_qkv_kernel(const float* part, long long plane, int ksplit, int ldo, int c0,
                               int mb, RowMap rows, int Hq, int Hkv, int d, const float2* rope,
                               __nv_bfloat16* q, __nv_bfloat16* arena, long long k_off,
                               long long v_off, int cap) {
  const int half = d / 2;
  const int heads = Hq + 2 * Hkv;
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)mb * heads * half) return;
  const int t = (int)(idx / (heads * half));
  const int rem = (int)(idx % (heads * half));
  const int hd = rem / half, j = rem % half;
  const int i = c0 + t;
  const long long col = (long long)hd * d + j;
  const float x1 = split_sum(part, plane, ksplit, (long long)t * ldo + col);
  const float x2 = split_sum(part, plane, ksplit, (long long)t * ldo + col + half);
  const int store = rows.P + i;
  if (hd < Hq + Hkv) {
    const float2 cs = rope[(long long)i * half + j];
    const float y1 = x1 * cs.x - x2 * cs.y;
    const float y2 = x2 * cs.x + x1 * cs.y;
    if (hd < Hq) {
      const int G = Hq / Hkv;
      __nv_bfloat16* dst = q + (((long long)(hd / G) * rows.m + i) * G + hd % G) * d;
      dst[j] = __float2bfloat16_rn(y1);
      dst[j + half] = __float2bfloat16_rn(y2);
    } else {
      __nv_bfloat16* dst = arena + k_off + ((long long)(hd - Hq) * cap + store) * d;
      dst[j] = __float2bfloat16_rn(y1);
      dst[j + half] = __float2bfloat16_rn(y2);
    }
  } else {
    // V is kept transposed in the slot: [Hkv][d][capacity]
    __nv_bfloat16* dst = arena + v_off + (long long)(hd - Hq - Hkv) * d * cap + store;
    dst[(long long)j * cap] = __float2bfloat16_rn(x1);
    dst[(long long)(j + half) * cap] = __float2bfloat16_rn(x2);
  }
}

// One CTA per token row: h += sum of the split partials (fixed split order),
// then RMSNorm of the new row for the next projection, or the bf16 output.
// float4 accesses; the row stays in registers between the two passes.
template <int V>  // float4 per thread (H <= 4 * 256 * V)
__global__ void __launch_bounds__(256) epi_resid_kernel(const float* part, long long plane, int ksplit,
                                                        int ldo, int c0, int H, float* h,
                                                        const __nv_bfloat16* gain, float eps,
                                                        __nv_bfloat16* a_out, __nv_bfloat16* final_out) {
  __shared__ float red[32];
  const int t = blockIdx.x;
  const long long i = c0 + t;
  const int H4 = H >> 2;
  float4 v[V];
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < V; ++u) {
    const int k4 = threadIdx.x + u * 256;
    if (k4 < H4) {
      float4 acc = reinterpret_cast<const float4*>(h + i * H)[k4];
      const float4* pp = reinterpret_cast<const float4*>(part + (long long)t * ldo) + k4;
      for (int s = 0; s < ksplit; ++s) {
        const float4 q = pp[s * (plane >> 2)];
        acc.x += q.x; acc.y += q.y; acc.z += q.z; acc.w += q.w;
      }
      reinterpret_cast<float4*>(h + i * H)[k4] = acc;
      ss += acc.x * acc.x + acc.y * acc.y + acc.z * acc.z + acc.w * acc.w;
      v[u] = acc;
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
      const int k4 = threadIdx.x + u * 256;
      if (k4 < H4) {
        const uint2 gw = reinterpret_cast<const uint2*>(gain)[k4];
        const __nv_bfloat162 g01 = *reinterpret_cast<const __nv_bfloat162*>(&gw.x);
        const __nv_bfloat162 g23 = *reinterpret_cast<const __nv_bfloat162*>(&gw.y);
        uint2 o;
        o.x = dev::pack_bf16x2(v[u].x * rs * __bfloat162float(g01.x), v[u].y * rs * __bfloat162float(g01.y));
        o.y = dev::pack_bf16x2(v[u].z * rs * __bfloat162float(g23.x), v[u].w * rs * __bfloat162float(g23.y));
        reinterpret_cast<uint2*>(a_out + i * H)[k4] = o;
      }
    }
  }
}

__global__ void epi_swiglu_kernel(const float* part, long long plane, int ksplit, int ldo, int c0,
                                  int mb, int F, __nv_bfloat16* z) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)mb * F) return;
  const int t = (int)(idx / F), n = (int)(idx % F);
  const float g = split_sum(part, plane, ksplit, (long long)t * ldo + n);
  const float u = split_sum(part, plane, ksplit, (long long)t * ldo + F + n);
  const float sg = g / (1.f + expf(-g));
  z[(long long)(c0 + t) * F + n] = __float2bfloat16_rn(sg * u);
}

__global__ void epi_cast_kernel(const float* part, long long plane, int ksplit, int ldo, int c0,
                                int mb, int N, __nv_bfloat16* out) {
  const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (long long)mb * N) return;
  const int t = (int)(idx / N), n = (int)(idx % N);
  out[(long long)(c0 + t) * N + n] =
      __float2bfloat16_rn(split_sum(part, plane, ksplit, (long long)t * ldo + n));
}

inline unsigned blocks_for(long long n, int threads) { return (unsigned)((n + threads - 1) / threads); }

}  // namespace

cudaError_t launch_rope_table(const RowMap& rows, int d, float theta, float2* table, cudaStream_t st) {
  const long long n = (long long)rows.m * (d / 2);
  rope_table_kernel<<<blocks_for(n, 256), 256, 0, st>>>(rows, d, (double)theta, table);
  return cudaGetLastError();
}

cudaError_t launch_embed(const __nv_bfloat16* hidden, int m, int H, const __nv_bfloat16* gain,
                         float eps, float* h, __nv_bfloat16* a, cudaStream_t st) {
  embed_kernel<<<m, 256, 0, st>>>(hidden, H, gain, eps, h, a);
  return cudaGetLastError();
}

cudaError_t launch_epi_qkv(const float* part, long long plane, int ksplit, int ldo, int c0, int mb,
                           const RowMap& rows, int Hq, int Hkv, int d, const float2* rope,
                           __nv_bfloat16* q, __nv_bfloat16* arena, long long k_off,
                           long long v_off, int cap, cudaStream_t st) {
  const long long n = (long long)mb * (Hq + 2 * Hkv) * (d / 2);
  epi_qkv_kernel<<<blocks_for(n, 256), 256, 0, st>>>(part, plane, ksplit, ldo, c0, mb, rows, Hq,
                                                     Hkv, d, rope, q, arena, k_off, v_off, cap);
  return cudaGetLastError();
}

cudaError_t launch_epi_resid(const float* part, long long plane, int ksplit, int ldo, int c0,
                             int mb, int H, float* h, const __nv_bfloat16* gain, float eps,
                             __nv_bfloat16* a_out, __nv_bfloat16* final_out, cudaStream_t st) {
  const int v = (H / 4 + 255) / 256;
  if (v <= 2)
    epi_resid_kernel<2><<<mb, 256, 0, st>>>(part, plane, ksplit, ldo, c0, H, h, gain, eps, a_out, final_out);
  else if (v <= 4)
    epi_resid_kernel<4><<<mb, 256, 0, st>>>(part, plane, ksplit, ldo, c0, H, h, gain, eps, a_out, final_out);
  else if (v <= 8)
    epi_resid_kernel<8><<<mb, 256, 0, st>>>(part, plane, ksplit, ldo, c0, H, h, gain, eps, a_out, final_out);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_epi_swiglu(const float* part, long long plane, int ksplit, int ldo, int c0,
                              int mb, int F, __nv_bfloat16* z, cudaStream_t st) {
  epi_swiglu_kernel<<<blocks_for((long long)mb * F, 256), 256, 0, st>>>(part, plane, ksplit, ldo,
                                                                         c0, mb, F, z);
  return cudaGetLastError();
}

cudaError_t launch_epi_cast(const float* part, long long plane, int ksplit, int ldo, int c0,
                            int mb, int N, __nv_bfloat16* out, cudaStream_t st) {
  epi_cast_kernel<<<blocks_for((long long)mb * N, 256), 256, 0, st>>>(part, plane, ksplit, ldo, c0,
                                                                      mb, N, out);
  return cudaGetLastError();
}

}  // namespace kvr
