// m-row batched GEMV: Y[t][n] = sum_k X[t][k] * W[n][k] for up to 32 token rows,
// each weight byte read from HBM once for all rows, with the projection's
// epilogue applied in the same launch.
//
// thinkspread, "The economics of speculative decoding" (cost model): the m
// verify rows run as one batched GEMV that streams each weight a single time
// for all of them, so an extra row costs far less than a full weight read.
//
// int4 group-32 path (the hot one).  A CTA owns a 128-row weight tile and a
// range of 256-input k-steps.  One producer warp streams, per k-step, a
// 128 x 128-byte int4 tile (128B-swizzled), its 128 x 8 fp16 scales and the
// 8*NT x 256 bf16 activation tile through TMA into a multi-stage
// shared-memory ring guarded by mbarriers.  Eight consumer warps each own 16
// weight rows:
//   * one 32-bit shared load per row gives a thread the eight 4-bit codes it
//     needs for the two m16n8k16 fragments of one 32-input group (the byte
//     layout of include/kvr.h is chosen for this);
//   * codes become exact bf16 integers (code+8 OR'd into the mantissa of 128.0,
//     minus 136);
//   * the unscaled group product sum_k code*x runs on the tensor cores with an
//     fp32 accumulator, and the fp16 group scale is applied afterwards in fp32:
//     acc += scale * group_sum.  The weight is therefore exactly code*scale,
//     never rounded to bf16.  (K-quant codes stay biased, 128 + q: the offset
//     folds into the sub-block's min term, which is formed anyway.)
// Plain CUDA-core FMAs would need 32*m FMAs per 16 weight bytes, more than the
// SM issues at HBM rate once m > 2; the tensor cores keep the kernel HBM-bound.
//
// Split k-steps: each CTA writes its fp32 partial tile, and the last CTA of
// the tile to arrive (an arrival counter per tile) adds the splits in split
// order -- the result does not depend on which CTA finishes last -- and runs
// the epilogue on the tile in shared memory:
//   * QKV: a tile is one head (d = 128) or two (d = 64), so each rotate-half
//     pair (j, j + d/2) is in the tile: RoPE at the row's position, bf16,
//     q to the KV-head-major q buffer, K rows and V^T columns to the slot
//     (goinfer "What goinfer does": one key and one value row per token and layer);
//   * Resid (applied as the contributions are added, with the residual row
//     loaded alongside them): h += y in fp32, and on the last layer out = bf16(h)
//     (the RMSNorm that follows needs the whole row, which no tile has: a
//     one-row-per-CTA launch forms it);
//   * Swiglu: the tile holds gate rows n0..n0+63 and the same up rows, so
//     z = bf16(silu(g) * u) is local to the tile;
//   * Cast: out = bf16(y) (attention-only layers);
//   * Argmax: per token, the tile's largest logit and its row (the LM head of
//     greedy verification; a small launch reduces the tiles).
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kConsumerWarps = kGemvRows / 16;   // 8
constexpr int kConsumers = kConsumerWarps * 32;  // 256
constexpr int kThreads = kConsumers + 32;
constexpr int kWTileBytes = kGemvRows * 128;       // 16 KB
constexpr int kSTileBytes = kGemvRows * 16;        // 2 KB
constexpr int kTileLd = kGemvRows + 4;             // fp32 result tile row stride (bank spread)

template <int NT>
struct GemvCfg {
  static constexpr int kXRows = 8 * NT;
  static constexpr int kXBoxBytes = kXRows * 128;             // one 64-input box
  static constexpr int kXTileBytes = 4 * kXBoxBytes;          // 256 inputs
  static constexpr int kStageBytes = kWTileBytes + kXTileBytes + kSTileBytes;
  static constexpr int kStages = 4;
  static constexpr int kSmem = kStages * kStageBytes + 1024;  // + alignment slack
  // the result tile reuses stage 0 once every stage has been consumed
  static_assert(kXRows * kTileLd * 4 <= kStageBytes, "result tile must fit in one stage");
};

// 8 4-bit fields of one 32-bit word -> 4 bf16x2 registers holding field - OFF
// (OFF = 8: the signed int4 code; 0: the unsigned K-quant code).
// Register i holds fields i (low half) and i+4 (high half).
// 8 4-bit fields of one 32-bit word -> 4 bf16x2 registers holding 128 + field
// (exact bf16 integers).  Register i holds fields i (low half) and i+4 (high
// half).
__device__ __forceinline__ void biased_word(uint32_t w, uint32_t r[4]) {
  const uint32_t magic = 0x43004300u;  // bf16 128.0 in both halves
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r[i]) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(magic));
}

// the same fields as signed int4 codes: 128 + field - 136 = code
__device__ __forceinline__ void code_word(uint32_t w, uint32_t r[4]) {
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
  biased_word(w, r);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 h = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&r[i]), bias);
    r[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// K-quant record (16 bytes: fp16 d, fp16 dmin, sixteen 6-bit fields at bits 6f
// of the little-endian 96-bit string in words y, z, w): (d*sc_g, dmin*mn_g)
__device__ __forceinline__ uint32_t q4k_field(const uint4& r, int f) {
  const int p = 6 * f, word = p >> 5, off = p & 31;
  const uint32_t lo = word == 0 ? r.y : (word == 1 ? r.z : r.w);
  const uint32_t hi = word == 0 ? r.z : r.w;
  return (off > 26 && word < 2 ? __funnelshift_r(lo, hi, off) : lo >> off) & 63u;
}

// (a, c) = (d*sc_g, 128*d*sc_g + dmin*mn_g): with the biased codes 128 + q on
// the tensor cores, sum(w x) = a * sum((128 + q) x) - c * sum(x)
__device__ __forceinline__ float2 q4k_ab(const uint4& r, int g) {
  const float d = __half2float(__ushort_as_half((unsigned short)(r.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(r.x >> 16)));
  const float a = d * (float)q4k_field(r, g);
  return make_float2(a, fmaf(128.f, a, dmin * (float)q4k_field(r, 8 + g)));
}

// barrier of the eight consumer warps (the producer warp has left)
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// ---------------------------------------------------------------- epilogues
// ct: the tile's fp32 results [token][kTileLd] for tokens < p.mb

// rope_s: the pass's rows of the RoPE table, [token][d/2] (staged in shared
// memory at the start of the launch)
__device__ __forceinline__ void epi_qkv(const GemvParams& p, const GemvSeg& seg, int s, int row0,
                                        const float* ct, const float2* rope_s, int tid) {
  const int d = p.d, half = d >> 1;
  const int nv = min(kGemvRows, seg.N - row0);
  const int hd0 = row0 / d;
  if (s < 2) {
    const int npairs = nv >> 1;
    const int G = p.Hq / p.Hkv;
    for (int idx = tid; idx < p.mb * npairs; idx += kConsumers) {
      const int t = idx / npairs, pr = idx % npairs;
      const int hh = pr / half, j = pr % half;
      const int col = hh * d + j;
      const float x1 = ct[t * kTileLd + col];
      const float x2 = ct[t * kTileLd + col + half];
      const int i = p.c0 + t;
      const float2 cs = rope_s[t * half + j];
      const float y1 = x1 * cs.x - x2 * cs.y;
      const float y2 = x2 * cs.x + x1 * cs.y;
      const int hd = hd0 + hh;
      __nv_bfloat16* dst =
          s == 0 ? p.q + q_row(p.rows, i, hd / G, hd % G, G, p.Hq) * d
                 : p.arena + p.k_off + row_slot(p.rows, i) * p.slot_stride +
                       ((long long)hd * p.cap + row_store(p.rows, i)) * d;
      dst[j] = __float2bfloat16_rn(y1);
      dst[j + half] = __float2bfloat16_rn(y2);
    }
  } else {
    // V^T: row (head, element) of the slot holds consecutive positions
    for (int idx = tid; idx < p.mb * nv; idx += kConsumers) {
      const int t = idx % p.mb, col = idx / p.mb;
      const int hd = hd0 + col / d, e = col % d;
      const int i = p.c0 + t;
      p.arena[p.v_off + row_slot(p.rows, i) * p.slot_stride + ((long long)hd * d + e) * p.cap +
              row_store(p.rows, i)] = __float2bfloat16_rn(ct[t * kTileLd + col]);
    }
  }
}

// Resid, one float4 of row i (columns row0 + c4 .. +3): h = h_old + y, and
// the final bf16 output on the last layer.
__device__ __forceinline__ void resid_apply(const GemvParams& p, int row0, long long i, int c4, float4 hv,
                                            const float4& y) {
  hv.x += y.x; hv.y += y.y; hv.z += y.z; hv.w += y.w;
  *reinterpret_cast<float4*>(p.h + i * p.H + row0 + c4) = hv;
  if (p.out) {
    uint2 o;
    o.x = dev::pack_bf16x2(hv.x, hv.y);
    o.y = dev::pack_bf16x2(hv.z, hv.w);
    *reinterpret_cast<uint2*>(p.out + i * p.ldout + row0 + c4) = o;
  }
}

__device__ __forceinline__ void epi_swiglu(const GemvParams& p, int row0, const float* ct, int tid) {
  const int nv = min(64, p.F - row0);
  for (int idx = tid; idx < p.mb * 64; idx += kConsumers) {
    const int t = idx >> 6, j = idx & 63;
    if (j >= nv) continue;
    const float g = ct[t * kTileLd + j], u = ct[t * kTileLd + 64 + j];
    const float sg = g / (1.f + expf(-g));
    p.z[(long long)(p.c0 + t) * p.F + row0 + j] = __float2bfloat16_rn(sg * u);
  }
}

__device__ __forceinline__ void epi_cast(const GemvParams& p, const GemvSeg& seg, int row0,
                                         const float* ct, int tid) {
  const int nv = min(kGemvRows, seg.N - row0);
  for (int idx = tid; idx < p.mb * kGemvRows; idx += kConsumers) {
    const int t = idx / kGemvRows, j = idx % kGemvRows;
    if (j >= nv) continue;
    p.out[(long long)(p.c0 + t) * p.ldout + seg.col0 + row0 + j] = __float2bfloat16_rn(ct[t * kTileLd + j]);
  }
}

// CTA owning unit u of the launch (units are tile-major: u = tile * ksteps + step)
__device__ __forceinline__ int unit_owner(long long u, int units, int ctas) {
  return (int)(((u + 1) * ctas - 1) / units);
}

constexpr int kMaxOwnTiles = 16;   // tiles one CTA may finish (host keeps it below)
constexpr int kConBatch = 8;       // contribution loads kept in flight by the reduction

// per token: the tile's largest logit and its row (lowest row on ties); warp w
// takes tokens w, w+8, ..., lane l rows l, l+32, l+64, l+96
__device__ __forceinline__ void epi_argmax(const GemvParams& p, const GemvSeg& seg, int tile, int row0,
                                           const float* ct, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  const int nv = min(kGemvRows, seg.N - row0);
  for (int t = warp; t < p.mb; t += kConsumerWarps) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int r = 0; r < kGemvRows / 32; ++r) {
      const int j = lane + 32 * r;
      const float v = j < nv ? ct[t * kTileLd + j] : -INFINITY;
      if (j < nv && (v > bv || (v == bv && j < bi))) { bv = v; bi = j; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if (lane == 0) p.best[(long long)(p.c0 + t) * p.tiles + tile] = make_float2(bv, (float)(row0 + bi));
  }
}

// segment and first weight row of a tile
template <bool kPair>
__device__ __forceinline__ int tile_seg(const GemvParams& p, int tile) {
  int s = 0;
  if (!kPair)
    while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile0) ++s;
  return s;
}
template <bool kPair>
__device__ __forceinline__ int tile_row0(const GemvParams& p, int tile, int s) {
  return kPair ? tile * 64 : (tile - p.seg[s].tile0) * kGemvRows;
}
// Producer (one lane): the weight and scale tiles of units [u0, u0 + nk) and
// their activation tiles through the stage ring.
template <int NT, bool kPair>
__device__ __forceinline__ void gemv_produce(const GemvParams& p, uint32_t base, uint64_t* full_bar,
                                             uint64_t* empty_bar, volatile int* abort_v, int u0, int nk) {
  using C = GemvCfg<NT>;
  for (int i = 0; i < p.nseg; ++i) {
    dev::prefetch_tmap(&p.seg[i].tw);
    dev::prefetch_tmap(&p.seg[i].ts);
  }
  if (kPair) {
    dev::prefetch_tmap(&p.seg[1].tw);
    dev::prefetch_tmap(&p.seg[1].ts);
  }
  dev::prefetch_tmap(&p.tx);
  const uint64_t pol = dev::policy_evict_first();
  auto load_w = [&](uint32_t sb, uint32_t fb, int u) {
    const int tile = u / p.ksteps, ks = u % p.ksteps;
    const int s = tile_seg<kPair>(p, tile);
    const int row0 = tile_row0<kPair>(p, tile, s);
    const uint32_t sc = sb + kWTileBytes + C::kXTileBytes;
    if (kPair) {
      dev::tma_load_2d_hint(sb, &p.seg[0].tw, ks * 128, row0, fb, pol);
      dev::tma_load_2d_hint(sb + kWTileBytes / 2, &p.seg[1].tw, ks * 128, row0, fb, pol);
      dev::tma_load_2d_hint(sc, &p.seg[0].ts, ks * 8, row0, fb, pol);
      dev::tma_load_2d_hint(sc + kSTileBytes / 2, &p.seg[1].ts, ks * 8, row0, fb, pol);
    } else {
      dev::tma_load_2d_hint(sb, &p.seg[s].tw, ks * 128, row0, fb, pol);
      dev::tma_load_2d_hint(sc, &p.seg[s].ts, ks * 8, row0, fb, pol);
    }
  };
  auto prefetch_w = [&](int u) {
    const int tile = u / p.ksteps, ks = u % p.ksteps;
    const int s = tile_seg<kPair>(p, tile);
    const int row0 = tile_row0<kPair>(p, tile, s);
    if (kPair) {
      dev::tma_prefetch_2d(&p.seg[0].tw, ks * 128, row0);
      dev::tma_prefetch_2d(&p.seg[1].tw, ks * 128, row0);
      dev::tma_prefetch_2d(&p.seg[0].ts, ks * 8, row0);
      dev::tma_prefetch_2d(&p.seg[1].ts, ks * 8, row0);
    } else {
      dev::tma_prefetch_2d(&p.seg[s].tw, ks * 128, row0);
      dev::tma_prefetch_2d(&p.seg[s].ts, ks * 8, row0);
    }
  };
  auto load_x = [&](uint32_t sb, uint32_t fb, int u) {
    const int ks = u % p.ksteps;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      dev::tma_load_2d(sb + kWTileBytes + j * C::kXBoxBytes, &p.tx, ks * kGemvKStep + 64 * j, p.c0, fb);
  };
  // Weights do not depend on earlier launches: fill the ring's weight and
  // scale tiles and pull the rest of this CTA's weights toward L2 before
  // waiting for the previous launch; the activations follow the wait.
  const int pre = nk < C::kStages ? nk : C::kStages;
  for (int it = 0; it < pre; ++it) {
    const uint32_t fb = dev::smem_u32(&full_bar[it]);
    dev::mbar_arrive_expect_tx(fb, C::kStageBytes);
    load_w(base + it * C::kStageBytes, fb, u0 + it);
  }
  for (int it = pre; it < nk; ++it) prefetch_w(u0 + it);
  dev::pdl_wait();
  for (int it = 0; it < pre; ++it)
    load_x(base + it * C::kStageBytes, dev::smem_u32(&full_bar[it]), u0 + it);
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
    load_w(sb, fb, u0 + it);
    load_x(sb, fb, u0 + it);
    ++issued;
  }
  // never leave the CTA with copies in flight: wait for the last use of
  // every stage that was filled, all within one bounded wait
  const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
  for (int st = 0; st < C::kStages && st < issued; ++st) {
    const int last = ((issued - 1 - st) / C::kStages) * C::kStages + st;
    dev::mbar_wait_until(dev::smem_u32(&full_bar[st]), (uint32_t)(last / C::kStages) & 1, deadline);
  }
}

// Consumers (8 warps, tid 0..255): units [u0, u0 + nk) into acc; at the end
// of each tile's run of units, seg_end(tile, acc, ok, last) takes the
// accumulators (and zeroes them).  A wait that gives up marks the CTA aborted;
// from then on the warps skip the work and the waits.  Returns ok.
template <int NT, int FMT, class SegEnd>
__device__ __forceinline__ bool gemv_consume(const GemvParams& p, uint32_t base, uint64_t* full_bar,
                                             uint64_t* empty_bar, volatile int* abort_v, float2* q4k_tab,
                                             int u0, int nk, float (&acc)[NT][4], SegEnd&& seg_end) {
  using C = GemvCfg<NT>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2;          // fragment row 0..7
  const int c = lane & 3;           // fragment column pair
  const int rho0 = warp * 16 + r;   // tile rows of this thread: rho0 and rho0+8
  const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
  bool ok = true;                   // warp-uniform
  for (int it = 0; it < nk; ++it) {
    const int st = it % C::kStages;
    const uint32_t use = (uint32_t)(it / C::kStages);
    if (ok) {
      const bool got = dev::mbar_wait(dev::smem_u32(&full_bar[st]), use & 1, p.status) && !*abort_v;
      ok = __all_sync(0xffffffffu, got);
      if (!ok && lane == 0) *abort_v = 1;
    }
    if (ok) {
      const uint32_t wt = base + st * C::kStageBytes;
      const uint32_t xt = wt + kWTileBytes;
      const uint32_t stile = xt + C::kXTileBytes;
      if constexpr (FMT == kFmtQ4K) {
        // one superblock per row and stage: the warp decodes (a, c) of its 16
        // rows x 8 sub-blocks once, then per sub-block
        //   acc += a * sum((128 + q) x) - c * sum(x)
        // with both sums on the tensor cores (128 + q exact in bf16, A = 1 for sum(x))
        float2* tab = q4k_tab + warp * 128;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int idx = lane + 32 * k;
          tab[idx] = q4k_ab(dev::lds128(stile + (warp * 16 + (idx >> 3)) * 16), idx & 7);
        }
        __syncwarp();
        const uint32_t one2 = 0x3F803F80u;   // bf16 1.0 in both halves
        const uint32_t a_one[4] = {one2, one2, one2, one2};
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint32_t w0 = dev::lds32(wt + dev::swz128(rho0, g) + 4 * c);
          const uint32_t w1 = dev::lds32(wt + dev::swz128(rho0 + 8, g) + 4 * c);
          uint32_t q0[4], q1[4];
          biased_word(w0, q0);
          biased_word(w1, q1);
          const uint32_t a_lo[4] = {q0[0], q1[0], q0[1], q1[1]};
          const uint32_t a_hi[4] = {q0[2], q1[2], q0[3], q1[3]};
          const float2 ab0 = tab[r * 8 + g], ab1 = tab[(r + 8) * 8 + g];
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const int n = t * 8 + (lane & 7);
            const int q = lane >> 3;
            const int box = g >> 1;
            const int chunk = 4 * (g & 1) + q;
            uint32_t b0, b1, b2, b3;
            dev::ldmatrix_x4(xt + box * C::kXBoxBytes + dev::swz128(n, chunk), b0, b1, b2, b3);
            float s1[4], s0[4];
            dev::mma_bf16_16816(s1, a_lo, b0, b1, zero4);
            dev::mma_bf16_16816(s1, a_hi, b2, b3, s1);
            dev::mma_bf16_16816(s0, a_one, b0, b1, zero4);
            dev::mma_bf16_16816(s0, a_one, b2, b3, s0);
            acc[t][0] = fmaf(ab0.x, s1[0], fmaf(-ab0.y, s0[0], acc[t][0]));
            acc[t][1] = fmaf(ab0.x, s1[1], fmaf(-ab0.y, s0[1], acc[t][1]));
            acc[t][2] = fmaf(ab1.x, s1[2], fmaf(-ab1.y, s0[2], acc[t][2]));
            acc[t][3] = fmaf(ab1.x, s1[3], fmaf(-ab1.y, s0[3], acc[t][3]));
          }
        }
      } else {
        // (removing the offset with two extra MMAs instead of the subtraction
        // measured slower here: the MMA issue, not the ALU, is the tighter limit)
        const uint4 sc0 = dev::lds128(stile + rho0 * 16);
        const uint4 sc1 = dev::lds128(stile + (rho0 + 8) * 16);
        const __half* s0h = reinterpret_cast<const __half*>(&sc0);
        const __half* s1h = reinterpret_cast<const __half*>(&sc1);
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint32_t w0 = dev::lds32(wt + dev::swz128(rho0, g) + 4 * c);
          const uint32_t w1 = dev::lds32(wt + dev::swz128(rho0 + 8, g) + 4 * c);
          uint32_t q0[4], q1[4];
          code_word(w0, q0);
          code_word(w1, q1);
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
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(dev::smem_u32(&empty_bar[st]));
    }
    const int u = u0 + it;
    if (u % p.ksteps == p.ksteps - 1 || it == nk - 1) seg_end(u / p.ksteps, acc, ok, it == nk - 1);
  }
  return ok;
}

// Stream-K: a CTA takes an equal run of (tile, k-step) units of the whole
// launch (the host sizes the grid to one resident wave: two CTAs per SM for
// up to 16 tokens, one beyond).
template <int NT, int EPI, int FMT>
__global__ void __launch_bounds__(kThreads, NT == 4 ? 1 : 2) gemv_int4_kernel(const __grid_constant__ GemvParams p) {
  using C = GemvCfg<NT>;
  constexpr bool kPair = EPI == kGemvEpiSwiglu;   // tile = 64 gate rows + 64 up rows
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ int abort_flag;
  __shared__ int n_own;
  __shared__ int own_tiles[kMaxOwnTiles];
  // K-quant: per warp and stage, (d*sc, dmin*mn) of its 16 rows x 8 sub-blocks
  __shared__ float2 q4k_tab[FMT == kFmtQ4K ? kConsumerWarps * 128 : 1];
  // QKV up to 8 tokens: the rows' (cos, sin), d <= 128 (more rows would cost
  // the second CTA per SM its shared memory; they read the table directly)
  constexpr bool kRopeS = EPI == kGemvEpiQKV && NT == 1;
  __shared__ float2 rope_s[kRopeS ? C::kXRows * 64 : 1];
  volatile int* abort_v = &abort_flag;

  const uint32_t base = (dev::smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // this CTA's contiguous range of (tile, k-step) units
  const int units = p.tiles * p.ksteps;
  const int u0 = (int)((long long)blockIdx.x * units / p.ctas);
  const int u1 = (int)((long long)(blockIdx.x + 1) * units / p.ctas);
  const int nk = u1 - u0;

  dev::pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&full_bar[i]), 1);
      dev::mbar_init(dev::smem_u32(&empty_bar[i]), kConsumerWarps);
    }
    // a wait of this or an earlier launch has given up: the call has failed,
    // and the whole CTA leaves before it issues a copy
    *abort_v = dev::status_set(p.status) ? 1 : 0;
    n_own = 0;
    dev::fence_mbar_init();
  }
  __syncthreads();
  if (*abort_v) return;

  if (warp == kConsumerWarps) {
    if (lane == 0) gemv_produce<NT, kPair>(p, base, full_bar, empty_bar, abort_v, u0, nk);
    return;
  }

  dev::pdl_wait();                  // results are written below
  const int tid = threadIdx.x;      // 0..255 over the consumer warps
  if (kRopeS)   // off the epilogue's path: loaded while the activations arrive
    for (int idx = tid; idx < p.mb * (p.d >> 1); idx += kConsumers)
      rope_s[idx] = p.rope[(long long)p.c0 * (p.d >> 1) + idx];
  const int r = lane >> 2, c = lane & 3;
  const int rho0 = warp * 16 + r;
  float acc[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
  // end of this CTA's part of a tile: store it as one contribution (the
  // arrivals are counted once, after the loop)
  gemv_consume<NT, FMT>(p, base, full_bar, empty_bar, abort_v, q4k_tab, u0, nk, acc,
                        [&](int tile, float (&a)[NT][4], bool ok, bool) {
    const int first = unit_owner((long long)tile * p.ksteps, units, p.ctas);
    float* tp = p.part + ((long long)tile * p.maxc + (blockIdx.x - first)) * (kGemvMaxCols * kGemvRows);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = t * 8 + 2 * c + (e & 1);
        if (ok && tok < p.mb) tp[tok * kGemvRows + rho0 + (e >> 1) * 8] = a[t][e];
        a[t][e] = 0.f;
      }
  });
  // publish every contribution of this CTA, then count one arrival per tile
  // touched (one thread per tile); the last arrival owns the tile's epilogue.
  // The barrier orders every consumer's partial stores before the counting
  // thread's acquire-release add (release is cumulative); its acquire side,
  // passed on by the barriers below, orders the other CTAs' partials before
  // this CTA's reads of them.
  consumers_sync();
  {
    const int t_first = u0 / p.ksteps, t_last = (u1 - 1) / p.ksteps;
    const int tile = t_first + tid;
    if (tile <= t_last && !*abort_v) {
      const long long tu0 = (long long)tile * p.ksteps;
      const int ncon = unit_owner(tu0 + p.ksteps - 1, units, p.ctas) - unit_owner(tu0, units, p.ctas) + 1;
      const int done = dev::atom_add_acq_rel(p.counters + tile, 1) + 1;
      if (done == ncon) {
        p.counters[tile] = 0;   // ready for the next launch
        const int k = atomicAdd(&n_own, 1);
        if (k < kMaxOwnTiles) own_tiles[k] = tile;
      }
    }
  }
  consumers_sync();
  if (tid == 0 && *abort_v) n_own = 0;          // an aborted CTA finishes nothing

  // ----------------------- tiles this CTA finished last: reduce, then epilogue
  consumers_sync();                            // own_tiles visible
  float* ct = reinterpret_cast<float*>(smem_raw + (base - dev::smem_u32(smem_raw)));
  const int n_done = min(n_own, kMaxOwnTiles);
  for (int k = 0; k < n_done; ++k) {
    const int tile = own_tiles[k];
    const long long tu0 = (long long)tile * p.ksteps;
    const int first = unit_owner(tu0, units, p.ctas);
    const int ncon = unit_owner(tu0 + p.ksteps - 1, units, p.ctas) - first + 1;
    const int s = tile_seg<kPair>(p, tile);
    const int row0 = tile_row0<kPair>(p, tile, s);
    const int nv_h = EPI == kGemvEpiResid ? min(kGemvRows, p.H - row0) : 0;
    const float* t0p = p.part + (long long)tile * p.maxc * (kGemvMaxCols * kGemvRows);
    for (int idx = tid; idx < p.mb * (kGemvRows / 4); idx += kConsumers) {
      const int tok = idx / (kGemvRows / 4), r4 = (idx % (kGemvRows / 4)) * 4;
      const float* src = t0p + tok * kGemvRows + r4;
      // Resid: the residual row's float4 travels with the contributions
      float4 h_old = make_float4(0.f, 0.f, 0.f, 0.f);
      if (EPI == kGemvEpiResid && r4 < nv_h)
        h_old = __ldcg(reinterpret_cast<const float4*>(p.h + (long long)(p.c0 + tok) * p.H + row0 + r4));
      // all contributions in flight at once, then added in contributor order
      // (the sum does not depend on which CTA arrived last)
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < ncon; j0 += kConBatch) {
        float4 w[kConBatch];
#pragma unroll
        for (int j = 0; j < kConBatch; ++j)
          if (j0 + j < ncon)
            w[j] = __ldcg(reinterpret_cast<const float4*>(src + (long long)(j0 + j) * (kGemvMaxCols * kGemvRows)));
#pragma unroll
        for (int j = 0; j < kConBatch; ++j)
          if (j0 + j < ncon) {
            v.x += w[j].x; v.y += w[j].y; v.z += w[j].z; v.w += w[j].w;
          }
      }
      if (EPI == kGemvEpiResid) {   // epilogue in place: no trip through shared memory
        if (r4 < nv_h) resid_apply(p, row0, p.c0 + tok, r4, h_old, v);
      } else {
        *reinterpret_cast<float4*>(ct + tok * kTileLd + r4) = v;
      }
    }
    if (EPI == kGemvEpiResid) continue;
    consumers_sync();
    if (EPI == kGemvEpiQKV) epi_qkv(p, p.seg[s], s, row0, ct, kRopeS ? rope_s : p.rope + (long long)p.c0 * (p.d >> 1), tid);
    else if (EPI == kGemvEpiSwiglu) epi_swiglu(p, row0, ct, tid);
    else if (EPI == kGemvEpiArgmax) epi_argmax(p, p.seg[s], tile, row0, ct, tid);
    else epi_cast(p, p.seg[s], row0, ct, tid);
    consumers_sync();
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

namespace {
// resident CTAs per SM of each (NT, EPI, FMT) variant, from the occupancy API
int g_per_sm[3][5][2];
}  // namespace

int gemv_int4_per_sm(int nt, int epi, int fmt) {
  return g_per_sm[nt == 1 ? 0 : (nt == 2 ? 1 : 2)][epi][fmt == kFmtQ4K ? 1 : 0];
}

namespace {

template <int NT>
cudaError_t setup_nt() {
  void (*ks[10])(GemvParams) = {
      gemv_int4_kernel<NT, 0, kFmtInt4>, gemv_int4_kernel<NT, 1, kFmtInt4>, gemv_int4_kernel<NT, 2, kFmtInt4>,
      gemv_int4_kernel<NT, 3, kFmtInt4>, gemv_int4_kernel<NT, 4, kFmtInt4>, gemv_int4_kernel<NT, 0, kFmtQ4K>,
      gemv_int4_kernel<NT, 1, kFmtQ4K>, gemv_int4_kernel<NT, 2, kFmtQ4K>, gemv_int4_kernel<NT, 3, kFmtQ4K>,
      gemv_int4_kernel<NT, 4, kFmtQ4K>};
  const int ni = NT == 1 ? 0 : (NT == 2 ? 1 : 2);
  for (int i = 0; i < 10; ++i) {
    cudaError_t e = cudaFuncSetAttribute(ks[i], cudaFuncAttributeMaxDynamicSharedMemorySize, GemvCfg<NT>::kSmem);
    int n = 0;
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, ks[i], kThreads, GemvCfg<NT>::kSmem);
    if (e != cudaSuccess) return e;
    g_per_sm[ni][i % 5][i / 5] = n;
  }
  return cudaSuccess;
}

template <int NT, int FMT>
cudaError_t launch_fmt(const GemvParams& p, dim3 grid, cudaStream_t st) {
  switch (p.epi) {
    case kGemvEpiQKV: return launch_k(gemv_int4_kernel<NT, 0, FMT>, grid, kThreads, GemvCfg<NT>::kSmem, st, p);
    case kGemvEpiResid: return launch_k(gemv_int4_kernel<NT, 1, FMT>, grid, kThreads, GemvCfg<NT>::kSmem, st, p);
    case kGemvEpiSwiglu: return launch_k(gemv_int4_kernel<NT, 2, FMT>, grid, kThreads, GemvCfg<NT>::kSmem, st, p);
    case kGemvEpiCast: return launch_k(gemv_int4_kernel<NT, 3, FMT>, grid, kThreads, GemvCfg<NT>::kSmem, st, p);
    case kGemvEpiArgmax: return launch_k(gemv_int4_kernel<NT, 4, FMT>, grid, kThreads, GemvCfg<NT>::kSmem, st, p);
  }
  return cudaErrorInvalidValue;
}

template <int NT>
cudaError_t launch_nt(const GemvParams& p, dim3 grid, cudaStream_t st) {
  return p.fmt == kFmtQ4K ? launch_fmt<NT, kFmtQ4K>(p, grid, st) : launch_fmt<NT, kFmtInt4>(p, grid, st);
}

}  // namespace

cudaError_t gemv_setup() {
  cudaError_t e = setup_nt<1>();
  if (e == cudaSuccess) e = setup_nt<2>();
  if (e == cudaSuccess) e = setup_nt<4>();
  return e;
}

cudaError_t launch_gemv_int4(const GemvParams& p, int nt, cudaStream_t st) {
  const dim3 grid(p.ctas);
  switch (nt) {
    case 1: return launch_nt<1>(p, grid, st);
    case 2: return launch_nt<2>(p, grid, st);
    default: return launch_nt<4>(p, grid, st);
  }
}

cudaError_t launch_gemv_bf16(const GemvParams& p, int total_cols, cudaStream_t st) {
  const int blocks = (total_cols * 32 + 255) / 256;
  return launch_k(gemv_bf16_kernel, blocks, 256, 0, st, p, total_cols);
}

}  // namespace kvr
