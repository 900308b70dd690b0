// Causal grouped-query attention of the new rows over a slot's cached prefix
// plus the new rows themselves, split across the key axis.
//
// goinfer, "Turn nine in under half a second" ("The problem", "What goinfer
// does"): prefill cost grows with the conversation; the cached rows' K/V are
// kept, so the m new rows attend to them instead of recomputing them.
// OpenJev "Latency" ("What changed"): several questions resume from one
// checkpoint -- each row sees the shared state plus its own question's rows.
//
// One CTA = (row tile, key split, KV head).  All G = Hq/Hkv query heads of a
// KV head and all m tokens are packed as rows (row = token*G + head-in-group),
// so each K/V tile is read from HBM once per (tile, split) for every query
// head that uses it.  A producer warp streams 64-key K tiles and V^T tiles (V
// is stored transposed in the slot) through TMA (128B-swizzled) into a
// 3-stage mbarrier ring; each consumer warp owns 16 rows: S = Q K^T and
// O += P V run as bf16 m16n8k16 tensor-core fragments (ldmatrix from the
// swizzled tiles), the online softmax runs
// in fp32 registers in the log2 domain with quad shuffles.  With several
// splits, unnormalised partials (O, running max, running sum) are merged by
// attn_combine in a fixed split order.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

// KW > 1: KW consumer warps share one 16-row tile and take alternate key
// blocks (their online-softmax states are merged at the end), with a deeper
// ring so that every warp has a block in flight.
template <int D, int KW = 1>
struct AttnCfg {
  static constexpr int kHalves = D / 64;                 // 64-element TMA boxes per row
  static constexpr int kTileBytes = kAttnKeys * D * 2;   // one K tile ([64 keys][D]) or V^T tile ([D][64 keys])
  static constexpr int kStageBytes = 2 * kTileBytes;
  // key-parallel (one row tile, a split of a few blocks): enough stages for
  // every block of a typical split to be requested at once (7 x 32 KB fits)
  static constexpr int kStages = KW > 1 ? (D == 128 ? 7 : 8) : (D == 128 ? 3 : 4);
  static constexpr int kSmem = kStages * kStageBytes + 1024;
  static_assert(KW * (16 * D + 32) * 4 <= kStages * kStageBytes, "warp merge buffer fits the ring");
};

// The part of the call one CTA serves: the whole call, or in a batched
// launch the conversation owning its row tile.
struct AttnView {
  int P, m;          // cached prefix, rows
  int kbase, vtbase;
  int nsplit;
  int rt;            // row tile within the rows
  const __nv_bfloat16* q;
  __nv_bfloat16* o;
  float* opart;
  float2* ml;
};

template <int D>
__device__ __forceinline__ AttnView attn_view(const AttnParams& p, int bx) {
  AttnView v;
  if (p.n_conv == 0) {
    v.P = p.rows.P; v.m = p.rows.m; v.kbase = p.kbase; v.vtbase = p.vtbase; v.nsplit = p.nsplit;
    v.rt = bx; v.q = p.q; v.o = p.o; v.opart = p.opart; v.ml = p.ml;
    return v;
  }
  int b = 0;
  while (b + 1 < p.n_conv && bx >= p.conv[b + 1].tile0) ++b;
  const AttnConv& cv = p.conv[b];
  v.P = cv.P; v.m = cv.m; v.kbase = cv.kbase; v.vtbase = cv.vtbase; v.nsplit = cv.nsplit;
  v.rt = bx - cv.tile0;
  const long long qd = (long long)cv.tok0 * p.Hq * D;
  v.q = p.q + qd; v.o = p.o + qd;
  v.opart = p.opart + cv.part0; v.ml = p.ml + cv.part0 / D;
  return v;
}

// 2^x with the PTX approximate base-2 exponential (ex2.approx.ftz.f32; 2^-inf
// = 0): one instruction on the per-element softmax chain
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct RowInfo {
  int tok;      // token index within the view, -1 for padding rows
  int head;     // query head
  int pre;      // keys [0, pre) are the cached prefix
  int lo, hi;   // own-branch visible slot indices [lo, hi]
};

__device__ __forceinline__ RowInfo row_info(const AttnParams& p, const AttnView& v, int kv, int rho) {
  RowInfo ri;
  const int R = p.G * v.m;
  ri.pre = v.P;
  if (rho >= R) {
    ri.tok = -1; ri.head = 0; ri.lo = 1; ri.hi = 0;
    return ri;
  }
  ri.tok = rho / p.G;
  ri.head = kv * p.G + rho % p.G;
  const int b = p.n_conv ? 0 : row_branch(p.rows, ri.tok);
  ri.lo = v.P + (p.n_conv ? 0 : p.rows.off[b]);
  ri.hi = v.P + ri.tok;
  return ri;
}

__device__ __forceinline__ bool visible(const RowInfo& ri, int j) {
  return ri.tok >= 0 && (j < ri.pre || (j >= ri.lo && j <= ri.hi));
}

// One warp merges the key splits' (O, max, sum) partials of one (token, head)
// row: lane s holds split s's (max, sum) (lane s-32 split s for ns > 32), the
// split weights are broadcast with shuffles, and each lane accumulates D/32
// consecutive elements over the splits in split order, NS splits' slices in
// flight at a time.  rows: rows per split plane; rowidx: this row's index.
template <int D, int NS>
__device__ __forceinline__ void merge_splits(const float* opart, const float2* mlp, long long rows,
                                             long long rowidx, int ns, __nv_bfloat16* dst, int lane,
                                             bool o16) {
  constexpr int E = D / 32;
  static_assert(kMaxSplits <= 64, "two split records per lane");
  const float* src = opart + rowidx * D + lane * E;
  const long long sstride = rows * D;
  // the first batch is requested before the split weights are formed
  float v[NS][E];
  auto load = [&](int s0) {
#pragma unroll
    for (int j = 0; j < NS; ++j)
      if (s0 + j < ns) {
        if (E == 4) {
          const float4 x = __ldcg(reinterpret_cast<const float4*>(src + (s0 + j) * sstride));
          v[j][0] = x.x; v[j][1 % E] = x.y; v[j][2 % E] = x.z; v[j][3 % E] = x.w;
        } else {
          const float2 x = __ldcg(reinterpret_cast<const float2*>(src + (s0 + j) * sstride));
          v[j][0] = x.x; v[j][1 % E] = x.y;
        }
      }
  };
  load(0);
  const float2 ml0 = lane < ns ? __ldcg(mlp + lane * rows + rowidx) : make_float2(-INFINITY, 0.f);
  const float2 ml1 = lane + 32 < ns ? __ldcg(mlp + (lane + 32) * rows + rowidx) : make_float2(-INFINITY, 0.f);
  float M = fmaxf(ml0.x, ml1.x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w0 = ml0.x == -INFINITY ? 0.f : exp2f(ml0.x - M);
  const float w1 = ml1.x == -INFINITY ? 0.f : exp2f(ml1.x - M);
  float den = w0 * ml0.y + w1 * ml1.y;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s0 = 0; s0 < ns; s0 += NS) {
    if (s0 > 0) load(s0);
#pragma unroll
    for (int j = 0; j < NS; ++j)
      if (s0 + j < ns) {
        const int sp = s0 + j;
        const float w = __shfl_sync(0xffffffffu, sp < 32 ? w0 : w1, sp & 31);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] += w * v[j][e];
      }
  }
  const float inv = 1.f / den;
  dst += rowidx * D + lane * E;
#pragma unroll
  for (int e = 0; e < E; e += 2)
    *reinterpret_cast<uint32_t*>(dst + e) = dev::pack_act2(acc[e] * inv, acc[e + 1] * inv, o16);
}

template <int D, int RW, int KW>
__global__ void __launch_bounds__((RW * KW + 1) * 32) attn_kernel(const __grid_constant__ AttnParams p) {
  static_assert(KW == 1 || RW == 1, "key-parallel warps serve one row tile");
  using C = AttnCfg<D, KW>;
  constexpr int kCons = RW * KW;   // consumer warps
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int abort_flag;
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const AttnView v = attn_view<D>(p, blockIdx.x);
  const int split = blockIdx.y, kv = blockIdx.z;
  if (split >= v.nsplit) return;   // a batched launch: this conversation uses fewer splits
  const int R = p.G * v.m;
  const int row_lo = v.rt * 16 * RW;
  const int row_hi = min(R, row_lo + 16 * RW);        // exclusive
  const int last_tok = (row_hi - 1) / p.G;
  const int kend = v.P + last_tok + 1;                 // keys [0, kend) may be visible
  const int nb = (kend + kAttnKeys - 1) / kAttnKeys;
  const int b0 = (int)((long long)nb * split / v.nsplit);
  const int b1 = (int)((long long)nb * (split + 1) / v.nsplit);
  const int nblk = b1 - b0;

  dev::pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&full_bar[i]), 1);
      dev::mbar_init(dev::smem_u32(&empty_bar[i]), RW);
    }
    // a wait has given up earlier in the call: leave before any copy
    *abort_v = dev::status_set(p.status) ? 1 : 0;
    dev::fence_mbar_init();
  }
  __syncthreads();
  if (*abort_v) return;

  if (warp == kCons) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      dev::prefetch_tmap(&p.tkv);
      dev::prefetch_tmap(&p.tvt);
      // Blocks wholly inside the cached prefix were written by earlier calls:
      // load them before waiting for the launch that appends this call's K/V.
      int pre = 0;
      while (pre < nblk && pre < C::kStages && (b0 + pre + 1) * kAttnKeys <= v.P) {
        const uint32_t sb = base + pre * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&full_bar[pre]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        const int key0 = (b0 + pre) * kAttnKeys;
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h)
          dev::tma_load_2d(sb + h * (kAttnKeys * 128), &p.tkv, 64 * h, v.kbase + kv * p.cap + key0, fb);
        dev::tma_load_2d(sb + C::kTileBytes, &p.tvt, key0, v.vtbase + kv * D, fb);
        ++pre;
      }
      dev::pdl_wait();
      int issued = pre;
      for (int it = pre; it < nblk; ++it) {
        const int st = it % C::kStages;
        const uint32_t use = (uint32_t)(it / C::kStages);
        if (it >= C::kStages) {
          if (!dev::mbar_wait(dev::smem_u32(&empty_bar[st]), (use - 1) & 1, p.status) ||
              *abort_v) {
            *abort_v = 1;
            break;
          }
        }
        const uint32_t sb = base + st * C::kStageBytes;
        const uint32_t fb = dev::smem_u32(&full_bar[st]);
        dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
        const int key0 = (b0 + it) * kAttnKeys;
#pragma unroll
        for (int h = 0; h < C::kHalves; ++h) {
          dev::tma_load_2d(sb + h * (kAttnKeys * 128), &p.tkv, 64 * h, v.kbase + kv * p.cap + key0, fb);
        }
        // V^T tile: D rows (head elements) x 64 keys
        dev::tma_load_2d(sb + C::kTileBytes, &p.tvt, key0, v.vtbase + kv * D, fb);
        ++issued;
      }
      const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
      for (int st = 0; st < C::kStages && st < issued; ++st) {
        const int last = ((issued - 1 - st) / C::kStages) * C::kStages + st;
        dev::mbar_wait_until(dev::smem_u32(&full_bar[st]), (uint32_t)(last / C::kStages) & 1, deadline);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  dev::pdl_wait();   // q comes from the previous launch
  const int r = lane >> 2, c = lane & 3;
  const int kw = KW > 1 ? warp : 0;                    // key-parallel warp
  const int rho0 = row_lo + (KW > 1 ? 0 : warp) * 16 + r;
  const RowInfo ri0 = row_info(p, v, kv, rho0);
  const RowInfo ri1 = row_info(p, v, kv, rho0 + 8);

  // Q fragments (A operand of S = Q K^T), loaded once
  uint32_t qa[D / 16][4];
  {
    const __nv_bfloat16* q0 =
        ri0.tok >= 0 ? v.q + (((long long)kv * v.m + ri0.tok) * p.G + ri0.head % p.G) * D : nullptr;
    const __nv_bfloat16* q1 =
        ri1.tok >= 0 ? v.q + (((long long)kv * v.m + ri1.tok) * p.G + ri1.head % p.G) * D : nullptr;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int d0 = kk * 16 + 2 * c;
      qa[kk][0] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + d0) : 0u;
      qa[kk][1] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + d0) : 0u;
      qa[kk][2] = q0 ? *reinterpret_cast<const uint32_t*>(q0 + d0 + 8) : 0u;
      qa[kk][3] = q1 ? *reinterpret_cast<const uint32_t*>(q1 + d0 + 8) : 0u;
    }
  }

  float o[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY};
  float lrow[2] = {0.f, 0.f};
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};

  for (int it = kw; it < nblk; it += KW) {
    const int st = it % C::kStages;
    const uint32_t use = (uint32_t)(it / C::kStages);
    if (!dev::mbar_wait(dev::smem_u32(&full_bar[st]), use & 1, p.status) || *abort_v) {
      *abort_v = 1;
      break;
    }
    const uint32_t kt = base + st * C::kStageBytes;
    const uint32_t vt = kt + C::kTileBytes;
    const int key0 = (b0 + it) * kAttnKeys;

    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int q = lane >> 3;
        const int key = 8 * (2 * np + (q >> 1)) + (lane & 7);
        const int chunk = 2 * kk + (q & 1);
        uint32_t b0r, b1r, b2r, b3r;
        dev::ldmatrix_x4(kt + (chunk >> 3) * (kAttnKeys * 128) + dev::swz128(key, chunk & 7), b0r,
                         b1r, b2r, b3r);
        dev::mma_bf16_16816(s[2 * np], qa[kk], b0r, b1r, s[2 * np]);
        dev::mma_bf16_16816(s[2 * np + 1], qa[kk], b2r, b3r, s[2 * np + 1]);
      }
    }

    // mask, scale to log2 units, online softmax
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = key0 + 8 * nt + 2 * c + (e & 1);
        const bool vis = (e < 2) ? visible(ri0, j) : visible(ri1, j);
        const float v = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
        s[nt][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float corr[2], muse[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
      mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
      const float mnew = fmaxf(mrow[h], mx[h]);
      muse[h] = mnew == -INFINITY ? 0.f : mnew;
      corr[h] = ex2_approx(mrow[h] - muse[h]);
      mrow[h] = mnew;
      lrow[h] *= corr[h];
    }
#pragma unroll
    for (int i = 0; i < D / 8; ++i) {
      o[i][0] *= corr[0]; o[i][1] *= corr[0];
      o[i][2] *= corr[1]; o[i][3] *= corr[1];
    }
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float pv = ex2_approx(s[nt][e] - muse[e >> 1]);
        s[nt][e] = pv;
        lrow[e >> 1] += pv;
      }
    }

    // O += P V: P as the A operand (16 keys per k-step); V^T rows are head elements,
    // so plain ldmatrix of the V^T tile yields the B fragments
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      uint32_t pa[4];
      pa[0] = dev::pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
      pa[1] = dev::pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
      pa[2] = dev::pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
      pa[3] = dev::pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int q = lane >> 3;
        const int drow = 16 * dp + 8 * (q >> 1) + (lane & 7);
        const int chunk = 2 * ks + (q & 1);
        uint32_t b0r, b1r, b2r, b3r;
        dev::ldmatrix_x4(vt + dev::swz128(drow, chunk), b0r, b1r, b2r, b3r);
        dev::mma_bf16_16816(o[2 * dp], pa, b0r, b1r, o[2 * dp]);
        dev::mma_bf16_16816(o[2 * dp + 1], pa, b2r, b3r, o[2 * dp + 1]);
      }
    }
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[st]));
  }
  (void)zero4;

#pragma unroll
  for (int h = 0; h < 2; ++h) {
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
    lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
  }
  if constexpr (KW > 1) {
    // merge the KW warps' (O, max, sum) of the same rows in shared memory (the
    // ring is drained: every block was consumed); warp 0 writes the result
    asm volatile("bar.sync 1, %0;" ::"r"(kCons * 32) : "memory");
    float* mb = reinterpret_cast<float*>(smem_raw + (base - dev::smem_u32(smem_raw)));
    float* mine = mb + kw * (16 * D + 32);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = r + 8 * h;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(mine + row * D + 8 * i + 2 * c) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
      if (c == 0) {
        mine[16 * D + row] = mrow[h];
        mine[16 * D + 16 + row] = lrow[h];
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCons * 32) : "memory");
    // with p.counters the other warps stay for the merge of the splits below
    // (every warp then reaches its barriers, aborted or not)
    if (kw != 0 && !(p.counters && v.nsplit > 1)) return;
    if (kw == 0 && !*abort_v)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = r + 8 * h;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < KW; ++w) M = fmaxf(M, mb[w * (16 * D + 32) + 16 * D + row]);
      float sc[KW];
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < KW; ++w) {
        const float mw = mb[w * (16 * D + 32) + 16 * D + row];
        sc[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
        L += sc[w] * mb[w * (16 * D + 32) + 16 * D + 16 + row];
      }
#pragma unroll
      for (int i = 0; i < D / 8; ++i) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < KW; ++w) {
          const float2 x = *reinterpret_cast<const float2*>(mb + w * (16 * D + 32) + row * D + 8 * i + 2 * c);
          acc.x += sc[w] * x.x;
          acc.y += sc[w] * x.y;
        }
        o[i][2 * h] = acc.x;
        o[i][2 * h + 1] = acc.y;
      }
      mrow[h] = M;
      lrow[h] = L;
    }
  }
  if (KW == 1 && *abort_v) return;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const RowInfo& ri = h == 0 ? ri0 : ri1;
    if (kw != 0 || ri.tok < 0 || *abort_v) continue;
    const long long rowidx = (long long)ri.tok * p.Hq + ri.head;
    if (v.nsplit == 1) {
      const float inv = 1.f / lrow[h];
      __nv_bfloat16* dst = v.o + rowidx * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<uint32_t*>(dst + 8 * i + 2 * c) =
            dev::pack_act2(o[i][2 * h] * inv, o[i][2 * h + 1] * inv, p.o16);
    } else {
      const long long plane = (long long)v.m * p.Hq;
      float* dst = v.opart + ((long long)split * plane + rowidx) * D;
#pragma unroll
      for (int i = 0; i < D / 8; ++i)
        *reinterpret_cast<float2*>(dst + 8 * i + 2 * c) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
      if (c == 0) v.ml[split * plane + rowidx] = make_float2(mrow[h], lrow[h]);
    }
  }
  if constexpr (KW > 1) {
    // The last split to finish this (row tile, KV head) merges every split's
    // partials (split order, as the combine kernel does), the KW warps taking
    // alternate rows.  The barrier orders warp 0's partial stores before the
    // counting thread's acquire-release add; its acquire side, passed on by
    // the second barrier, orders the other splits' partials before the loads.
    if (!p.counters || v.nsplit == 1) return;
    __shared__ int last_split;
    asm volatile("bar.sync 1, %0;" ::"r"(kCons * 32) : "memory");
    if (threadIdx.x == 0) {   // an aborted CTA does not count: its row tile is left unmerged
      last_split = 0;
      if (!*abort_v) {
        int* ctr = p.counters + (long long)blockIdx.x * p.Hkv + kv;
        const int done = dev::atom_add_acq_rel(ctr, 1) + 1;
        last_split = done == v.nsplit;
        if (done == v.nsplit) *ctr = 0;   // ready for the next launch
      }
    }
    asm volatile("bar.sync 1, %0;" ::"r"(kCons * 32) : "memory");
    if (!last_split) return;
    const long long plane = (long long)v.m * p.Hq;
    for (int rho = row_lo + kw; rho < row_hi; rho += KW) {
      const RowInfo ri = row_info(p, v, kv, rho);
      if (ri.tok < 0) continue;
      merge_splits<D, 16>(v.opart, v.ml, plane, (long long)ri.tok * p.Hq + ri.head, v.nsplit, v.o, lane, p.o16);
    }
  }
}

// One warp per (token, head) row: merge the key splits' (O, max, sum)
// partials.  Lane s holds split s's (max, sum) (and lane s-32 split s for
// nsplit > 32); the split weights are broadcast with shuffles and each lane
// accumulates D/32 consecutive elements over the splits in split order, NS
// splits' loads in flight at a time.
template <int D, int NS>   // NS: split slices loaded per batch
__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ AttnParams p) {
  dev::pdl_trigger();
  dev::pdl_wait();
  const long long grow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);   // (token, head) of the call
  if (grow >= (long long)p.rows.m * p.Hq) return;
  // the row's partials: of the whole call, or of its conversation in a batch
  long long rows = (long long)p.rows.m * p.Hq, rowidx = grow;
  int ns = p.nsplit;
  const float* opart = p.opart;
  const float2* mlp = p.ml;
  if (p.n_conv) {
    const int tok = (int)(grow / p.Hq);
    int b = 0;
    while (b + 1 < p.n_conv && tok >= p.conv[b + 1].tok0) ++b;
    const AttnConv& cv = p.conv[b];
    ns = cv.nsplit;
    if (ns == 1) return;   // the attention kernel wrote this row itself
    rows = (long long)cv.m * p.Hq;
    rowidx = grow - (long long)cv.tok0 * p.Hq;
    opart += cv.part0;
    mlp += cv.part0 / D;
  }
  // row rowidx of the conversation's planes is row grow of the call's o
  merge_splits<D, NS>(opart, mlp, rows, rowidx, ns, p.o + (grow - rowidx) * D, threadIdx.x & 31, p.o16);
}

template <int D, int RW, int KW = 1>
cudaError_t launch_t(const AttnParams& p, cudaStream_t st) {
  const dim3 grid(p.row_tiles, p.nsplit, p.Hkv);
  return launch_k(attn_kernel<D, RW, KW>, grid, (RW * KW + 1) * 32, AttnCfg<D, KW>::kSmem, st, p);
}

template <int D>
cudaError_t setup_d() {
  cudaError_t e;
  e = cudaFuncSetAttribute(attn_kernel<D, 1, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<D, 4>::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(attn_kernel<D, 2, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<D>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(attn_kernel<D, 4, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnCfg<D>::kSmem);
}

}  // namespace

int attn_key_warps(int row_warps) { return row_warps == 1 ? 4 : 1; }

cudaError_t attn_setup() {
  cudaError_t e = setup_d<64>();
  if (e != cudaSuccess) return e;
  return setup_d<128>();
}

// one row tile (R <= 16): four key-parallel warps; more rows: 2 or 4 row warps
cudaError_t launch_attention(const AttnParams& p, int d, int row_warps, cudaStream_t st) {
  if (d == 128) {
    if (row_warps == 1) return launch_t<128, 1, 4>(p, st);
    if (row_warps == 2) return launch_t<128, 2>(p, st);
    return launch_t<128, 4>(p, st);
  }
  if (row_warps == 1) return launch_t<64, 1, 4>(p, st);
  if (row_warps == 2) return launch_t<64, 2>(p, st);
  return launch_t<64, 4>(p, st);
}

cudaError_t launch_attn_combine(const AttnParams& p, int d, cudaStream_t st) {
  const unsigned blocks = (unsigned)((p.rows.m * p.Hq + 7) / 8);
  // few splits (large m): a short batch keeps registers and occupancy; many
  // splits (small m): all of them in flight
  if (p.nsplit <= 4) {
    if (d == 128) return launch_k(attn_combine_kernel<128, 4>, blocks, 256, 0, st, p);
    return launch_k(attn_combine_kernel<64, 4>, blocks, 256, 0, st, p);
  }
  if (p.nsplit <= 8) {
    if (d == 128) return launch_k(attn_combine_kernel<128, 8>, blocks, 256, 0, st, p);
    return launch_k(attn_combine_kernel<64, 8>, blocks, 256, 0, st, p);
  }
  if (d == 128) return launch_k(attn_combine_kernel<128, 32>, blocks, 256, 0, st, p);
  return launch_k(attn_combine_kernel<64, 32>, blocks, 256, 0, st, p);
}

}  // namespace kvr
