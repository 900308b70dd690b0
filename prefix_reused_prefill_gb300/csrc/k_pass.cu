// The small-m suffix prefill as one persistent pass: every layer of the stack
// for up to 16 rows in a single cooperative launch, one CTA per SM.
//
// thinkspread, "The economics of speculative decoding" (cost model): a
// verify of m = k+1 rows reads every weight once for all of them, so at small
// m the call is a stream of weight bytes.  goinfer, "What goinfer does": the
// rows append one key and one value row per layer to their slot and attend to
// the slot's cached prefix plus themselves.
//
// Separate launches per projection leave the weight stream idle at every
// step boundary (a launch edge, the activations' first load, the split-K
// tail, the slowest CTA).  Here each CTA keeps one ring of shared-memory
// stages that a producer warp fills: it walks the whole call's schedule --
// its share of every projection's (tile, 256-input step) units and its
// attention item's 64-key blocks, layer after layer -- and issues the copy of
// each use as soon as its stage is free.  The weights of the next steps
// therefore stream while the consumers wait for the current step's inputs.
// The producer is a warp of its own: copies issued from inside a consumer's
// wait loop are issued late (that warp's other lanes sleep on the barrier,
// and the issuing lane moves on before the last consumer frees a stage), and
// the stream then runs at about 60% of the rate a free-running producer gets.
//
// Steps of a layer and what each waits for (counters in global memory that
// grow by one call's count per call, read with acquire loads):
//   QKV   x = bf16(RMSNorm(h) * g_attn) from h and its per-tile sums of
//         squares (the previous layer's down step, or the embedding);
//         epilogue: RoPE, q, the slot's K row and V^T column;
//   ATTN  (KV head, key split) items over the slot's 64-key blocks: S = Q K^T
//         and O += P V on tensor-core fragments with an online softmax; the
//         last split of a KV head to finish merges the splits in split order
//         into o.  Blocks that hold this call's rows wait for QKV;
//   O     x = o; epilogue h += y and the new rows' sums of squares per tile;
//   GU    x = bf16(RMSNorm(h) * g_ffn); tile = 64 gate + the same 64 up rows,
//         epilogue z = bf16(silu(g) * u);
//   DOWN  x = z; epilogue h += y (and the bf16 output on the last layer).
// Each projection is split stream-K over all CTAs as in the GEMV kernel: a
// CTA stores its partial tile, and the last contributor of a tile to arrive
// adds the partials in contributor order (the result does not depend on
// timing) and applies the epilogue.  The eight consumer warps share a unit,
// one 16-row group of the 128-row tile each, over all 256 inputs (nine warps
// leave 224 registers a thread).  The activations of a unit are staged by the
// consumers (bf16, swizzled as the GEMV's TMA tiles) one unit ahead of its
// weights.
//
// Every wait is bounded (1 s) and reports through the status word; a CTA that
// finds the word set stops, drains its copies and leaves.
#include "kvr_internal.cuh"

namespace kvr {

namespace {

constexpr int kWarps = 8;                     // consumer warps (one 16-row group of a tile each)
constexpr int kCons = kWarps * 32;
constexpr int kThreads = kCons + 64;          // the producer warp and the L2 prefetch warp
constexpr int kPfAhead = 16;                  // uses the L2 prefetch runs ahead of the copies
constexpr int kStage = 18 * 1024;             // int4 tile 16 KB + scales 2 KB, or one K / V^T tile
constexpr int kStages = 8;
// activations of a projection step, staged for up to kXArea / (4 * 1 KB * NT)
// units at a time: per unit four 64-input boxes of 8 * NT rows (GEMV layout)
constexpr int kXArea = 64 * 1024;
constexpr int kCtLd = kGemvRows + 4;          // tile buffer row stride (floats)
constexpr int kCtBytes = kPassRows * kCtLd * 4;
constexpr int kAttnD = 128;
constexpr int kMergeState = 16 * (kAttnD / 2) + 32;   // floats of one warp's state (half the head dims)
constexpr int kMergeBytes = 8 * kMergeState * 4;
// attention: up to two 16-row tiles keep four warp states plus their query
// rows; three or four tiles (one warp each) keep only the query rows
constexpr int kAttnWork = kMergeBytes + 2 * 16 * kAttnD * 2;
static_assert(kPassMaxAttnRows * kAttnD * 2 <= kAttnWork, "query rows of four tiles fit");
static_assert(kCtBytes <= kXArea, "the epilogue's tile buffer fits the staging area");
constexpr int kWork = (kXArea > kAttnWork ? kXArea : kAttnWork);
constexpr int kSmem = kStages * kStage + kWork + 1024;
constexpr int kMaxOwn = 16;                   // tiles one CTA may finish per projection
static_assert(kSmem <= 232448, "shared memory of one CTA");

constexpr int kPhQKV = 0, kPhAttn = 1, kPhO = 2, kPhGU = 3, kPhDown = 4;

// ------------------------------------------------------------ projection steps
struct Proj {
  int ph;
  int nseg;
  int tiles;
  int ksteps;
  bool pair;       // gate|up: tile = 64 gate rows + the same 64 up rows
  int t1, t2;      // QKV: first tile of k and of v
  int qd, kvd, N;  // QKV widths; other steps: the output rows
};

__device__ __forceinline__ Proj proj_of(const PassParams& p, int ph) {
  Proj j;
  j.ph = ph;
  j.pair = ph == kPhGU;
  j.qd = p.Hq * p.d;
  j.kvd = p.Hkv * p.d;
  j.t1 = j.t2 = 1 << 30;
  j.nseg = 1;
  if (ph == kPhQKV) {
    j.nseg = 3;
    j.t1 = (j.qd + kGemvRows - 1) / kGemvRows;
    j.t2 = j.t1 + (j.kvd + kGemvRows - 1) / kGemvRows;
    j.tiles = j.t2 + (j.kvd + kGemvRows - 1) / kGemvRows;
    j.ksteps = p.H / kGemvKStep;
    j.N = j.qd;
  } else if (ph == kPhO) {
    j.N = p.H;
    j.tiles = (p.H + kGemvRows - 1) / kGemvRows;
    j.ksteps = j.qd / kGemvKStep;
  } else if (ph == kPhGU) {
    j.N = p.F;
    j.tiles = (p.F + 63) / 64;
    j.ksteps = p.H / kGemvKStep;
  } else {
    j.N = p.H;
    j.tiles = (p.H + kGemvRows - 1) / kGemvRows;
    j.ksteps = p.F / kGemvKStep;
  }
  return j;
}

// segment of a tile (QKV: 0 q, 1 k, 2 v), its first weight row, its output
// rows and its PassLayer matrix
__device__ __forceinline__ int seg_of(const Proj& j, int tile) { return tile >= j.t2 ? 2 : (tile >= j.t1 ? 1 : 0); }
__device__ __forceinline__ int row0_of(const Proj& j, int tile, int s) {
  return j.pair ? tile * 64 : (tile - (s == 0 ? 0 : (s == 1 ? j.t1 : j.t2))) * kGemvRows;
}
__device__ __forceinline__ int rows_of(const Proj& j, int s) { return j.ph == kPhQKV ? (s == 0 ? j.qd : j.kvd) : j.N; }
__device__ __forceinline__ int mat_of(const Proj& j, int s) {
  return j.ph == kPhQKV ? s : (j.ph == kPhO ? 3 : (j.ph == kPhGU ? 4 + s : 6));
}
// A projection's units are split over its first min(ctas, units) CTAs, each
// an equal run of at least one unit, so the CTAs that touch a tile are
// consecutive and each contributes one partial.
__device__ __forceinline__ int proj_ctas(int units, int ctas) { return units < ctas ? units : ctas; }
// this CTA's units [u0, u1) of a projection with `units` units
__device__ __forceinline__ void unit_range(int units, int ctas, int cta, int& u0, int& u1) {
  const int n = proj_ctas(units, ctas);
  u0 = cta < n ? (int)((long long)cta * units / n) : units;
  u1 = cta < n ? (int)((long long)(cta + 1) * units / n) : units;
}
__device__ __forceinline__ int owner_of(long long u, int units, int ctas) {
  const int n = proj_ctas(units, ctas);
  return (int)(((u + 1) * n - 1) / units);
}

// ------------------------------------------------------------ attention items
struct Item {
  bool any;
  int kv, split, b0, b1;
};
__device__ __forceinline__ Item item_of(const PassParams& p, int cta) {
  Item it;
  it.any = cta < p.Hkv * p.nsplit;
  it.kv = it.any ? cta / p.nsplit : 0;
  it.split = it.any ? cta % p.nsplit : 0;
  it.b0 = (int)((long long)p.nb * it.split / p.nsplit);
  it.b1 = it.any ? (int)((long long)p.nb * (it.split + 1) / p.nsplit) : it.b0;
  return it;
}

__device__ __forceinline__ int done_index(int layer, int ph) { return layer * kPassPhases + ph; }
__device__ __forceinline__ int done_count(const PassParams& p, int ph) {
  if (ph == kPhAttn) return p.Hkv;
  return proj_of(p, ph).tiles;
}

__device__ __forceinline__ int ld_acquire(const int* ptr) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}
__device__ __forceinline__ void red_release_add(int* ptr, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Polls of global words (the completion counters, the status word) are spaced
// in time: thousands of threads reading one L2 line back to back slow every
// other request that line's L2 slice serves, the weight copies included.
constexpr unsigned long long kPollNs = 4000;
constexpr unsigned kCountBackoffNs = 100;

// The first wait of a pass to give up records where in the status word:
// bit 0 set, the wait site in bits 1-3, a site detail (the counter index or
// the ring use) in bits 4-15 and the CTA in bits 16-30.
__device__ __forceinline__ int site_code(int site, int detail) {
  return kStatusTimeout | (site << 1) | ((detail & 0xFFF) << 4) | ((int)(blockIdx.x & 0x7FFF) << 16);
}
__device__ __forceinline__ void give_up(int* status, int* diag, int site, int detail, int seen) {
  const int code = site_code(site, detail);
  atomicCAS(status, 0, code);
  if (diag && blockIdx.x < kPassMaxCtas) {
    diag[2 * blockIdx.x] = code;
    diag[2 * blockIdx.x + 1] = seen;
  }
}
constexpr int kSiteConsCount = 2, kSiteConsRing = 4, kSiteProdRing = 5, kSiteProdCount = 6;

// An mbarrier phase wait of the pass: as dev::mbar_wait, with its site recorded
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, int* status, int* diag, int site, int detail) {
  if (dev::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = dev::globaltimer_ns();
  unsigned long long next_check = t0 + kPollNs;
  for (;;) {
    if (dev::mbar_try_wait(bar, parity)) return true;
    const unsigned long long t = dev::globaltimer_ns();
    if (t > next_check) {   // another wait may have given up (checked every few microseconds)
      if (dev::status_set(status)) return false;
      next_check = t + kPollNs;
    }
    if (t - t0 > kWaitLimitNs) {
      give_up(status, diag, site, detail, (int)parity);
      return false;
    }
  }
}

// (the non-aligned barrier forms: thread 0 reaches them from its own loops)
__device__ __forceinline__ void cons_sync() { asm volatile("barrier.sync 1, 256;" ::: "memory"); }

// Barrier of the CTA's warps that also ORs one flag over all of them: every
// thread gets the same answer, so a decision taken on it is uniform (the
// abort flag itself may be set by any warp at any time).
__device__ __forceinline__ bool cons_sync_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "barrier.red.or.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// 8 4-bit fields of one 32-bit word -> 4 bf16x2 registers holding the signed
// codes (field - 8, exact bf16 integers); register i holds fields i and i+4
__device__ __forceinline__ void codes_bf16(uint32_t w, uint32_t r[4]) {
  const __nv_bfloat162 bias = __floats2bfloat162_rn(136.0f, 136.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(v) : "r"(w >> (4 * i)), "r"(0x000F000Fu), "r"(0x43004300u));
    __nv_bfloat162 h = __hsub2(*reinterpret_cast<__nv_bfloat162*>(&v), bias);
    r[i] = *reinterpret_cast<uint32_t*>(&h);
  }
}

// ------------------------------------------------------------ shared state
struct Shared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  Item item;                              // this CTA's attention item
  int u0[kPassPhases], u1[kPassPhases];   // this CTA's units of each projection step
  unsigned issued;                        // uses the producer has issued
  int abort;
  int n_own;
  int own[kMaxOwn];
  float rscale[kPassRows];
  int merge_last;
};
__shared__ Shared sh;

// ============================================================== the producer
// Lane 0 of the producer warp walks the call's schedule of ring uses -- this
// CTA's units of every projection step and its attention item's key blocks
// (a K tile, then a V^T tile), layer after layer -- and issues the copy of
// each use as soon as its stage is free, so the weights of later steps stream
// while the consumers wait for a step's inputs.  Key blocks that hold this
// call's rows are issued once the layer's QKV step is complete, after a proxy
// fence, since the consumers' generic stores wrote them.  Everything that
// needs a division is worked out once per step; an issue only advances the
// step's (tile, k-step) cursor.
struct Cursor {
  int l, ph;              // step: layer, phase
  int k, n;               // index within the step's uses, their count
  int tile, ks, ksteps;
  int seg, seg_end, t2;   // QKV segment (0 q, 1 k, 2 v), its end tile, the first v tile
  int row0, rstep;        // weight row of the tile, rows from one tile to the next
  int wi;                 // PassLayer matrix of the segment (gate|up: 4 and 5)
  bool pair;
  const PassLayer* Ly;
  int kb, vb, b;          // attention: view rows of the layer's K and V^T, the block
};

__device__ __forceinline__ void cursor_enter(const PassParams& p, Cursor& c) {
  c.k = 0;
  if (c.ph == kPhAttn) {
    const Item& item = sh.item;
    c.n = 2 * (item.b1 - item.b0);
    c.b = item.b0;
    c.kb = p.kbase0 + c.l * 2 * p.Hkv * p.cap + item.kv * p.cap;
    c.vb = p.vtbase0 + c.l * 2 * p.Hkv * p.d + item.kv * p.d;
    return;
  }
  const Proj j = proj_of(p, c.ph);
  const int u0 = sh.u0[c.ph];
  c.n = sh.u1[c.ph] - u0;
  if (c.n <= 0) return;
  c.ksteps = j.ksteps;
  c.tile = u0 / j.ksteps;
  c.ks = u0 % j.ksteps;
  c.seg = seg_of(j, c.tile);
  c.t2 = j.t2;
  c.seg_end = c.seg == 0 ? j.t1 : (c.seg == 1 ? j.t2 : (1 << 30));
  c.row0 = row0_of(j, c.tile, c.seg);
  c.rstep = j.pair ? 64 : kGemvRows;
  c.pair = j.pair;
  c.wi = mat_of(j, c.seg);
  c.Ly = p.layers + c.l;
  for (int s = 0; s < (j.pair ? 2 : 1); ++s) {
    dev::prefetch_tmap(&c.Ly->tw[c.wi + s]);
    dev::prefetch_tmap(&c.Ly->ts[c.wi + s]);
  }
}

// advance a projection cursor past one use: the next k-step, the next tile,
// the next QKV segment
__device__ __forceinline__ void cursor_next_unit(Cursor& c) {
  if (++c.ks == c.ksteps) {
    c.ks = 0;
    c.row0 += c.rstep;
    if (++c.tile == c.seg_end) {
      ++c.seg;
      c.wi = c.seg;   // QKV: matrices 0, 1, 2
      c.row0 = 0;
      c.seg_end = c.seg == 1 ? c.t2 : (1 << 30);
      dev::prefetch_tmap(&c.Ly->tw[c.wi]);
      dev::prefetch_tmap(&c.Ly->ts[c.wi]);
    }
  }
}

// Wait (bounded) for an mbarrier phase on the producer's side: gives up when
// the consumers have aborted, when the status word is set, or after the limit.
__device__ __forceinline__ bool producer_wait(const PassParams& p, uint32_t bar, uint32_t parity, int detail) {
  if (dev::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = dev::globaltimer_ns();
  unsigned long long next_check = t0 + kPollNs;
  for (;;) {
    if (dev::mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&sh.abort)) return false;
    const unsigned long long t = dev::globaltimer_ns();
    if (t > next_check) {
      if (dev::status_set(p.status)) return false;
      next_check = t + kPollNs;
    }
    if (t - t0 > kWaitLimitNs) {
      give_up(p.status, p.diag, kSiteProdRing, detail, (int)parity);
      return false;
    }
  }
}

__device__ __noinline__ void producer(const PassParams& p, uint32_t ring) {
  const uint64_t pol = dev::policy_evict_first();
  dev::prefetch_tmap(&p.tkv);
  dev::prefetch_tmap(&p.tvt);
  Cursor c;
  c.l = 0;
  c.ph = 0;
  cursor_enter(p, c);
  int qkv_l = -1;   // last layer whose QKV step is known complete
  unsigned it = 0;  // uses issued
  bool live = true;
  while (live) {
    if (c.k >= c.n) {   // the step is exhausted: the next one
      if (++c.ph == kPassPhases) {
        c.ph = 0;
        if (++c.l == p.L) break;
      }
      cursor_enter(p, c);
      continue;
    }
    const int st = (int)(it % kStages);
    if (it >= (unsigned)kStages && !producer_wait(p, dev::smem_u32(&sh.empty[st]), ((it / kStages) - 1) & 1, (int)it))
      break;
    const uint32_t sb = ring + st * kStage;
    const uint32_t fb = dev::smem_u32(&sh.full[st]);
    if (c.ph == kPhAttn) {
      if ((c.b + 1) * kAttnKeys > p.rows.P && qkv_l < c.l) {
        // this block holds rows of this call, appended by the layer's QKV step
        const int* ctr = p.done + done_index(c.l, kPhQKV);
        const int target = (int)p.epoch * done_count(p, kPhQKV);
        const unsigned long long t0 = dev::globaltimer_ns();
        for (unsigned n = 0; ld_acquire(ctr) - target < 0; ++n) {
          __nanosleep(kCountBackoffNs);
          if (*reinterpret_cast<volatile int*>(&sh.abort) || ((n & 15u) == 15u && dev::status_set(p.status))) {
            live = false;
            break;
          }
          if (dev::globaltimer_ns() - t0 > kWaitLimitNs) {
            give_up(p.status, p.diag, kSiteProdCount, done_index(c.l, kPhQKV), ld_acquire(ctr));
            live = false;
            break;
          }
        }
        if (!live) break;
        fence_proxy_async_global();
        qkv_l = c.l;
      }
      dev::mbar_arrive_expect_tx(fb, kAttnKeys * kAttnD * 2);
      if ((c.k & 1) == 0) {
        const int kr = c.kb + c.b * kAttnKeys;
        dev::tma_load_2d(sb, &p.tkv, 0, kr, fb);
        dev::tma_load_2d(sb + kAttnKeys * 128, &p.tkv, 64, kr, fb);
      } else {
        dev::tma_load_2d(sb, &p.tvt, c.b * kAttnKeys, c.vb, fb);
        ++c.b;
      }
    } else {
      const CUtensorMap* tw = &c.Ly->tw[c.wi];
      const CUtensorMap* ts = &c.Ly->ts[c.wi];
      const int x = c.ks * 128, xs = c.ks * 8, y = c.row0;
      dev::mbar_arrive_expect_tx(fb, kStage);
      if (c.pair) {
        dev::tma_load_2d_hint(sb, tw, x, y, fb, pol);
        dev::tma_load_2d_hint(sb + 64 * 128, tw + 1, x, y, fb, pol);
        dev::tma_load_2d_hint(sb + 128 * 128, ts, xs, y, fb, pol);
        dev::tma_load_2d_hint(sb + 128 * 128 + 64 * 16, ts + 1, xs, y, fb, pol);
      } else {
        dev::tma_load_2d_hint(sb, tw, x, y, fb, pol);
        dev::tma_load_2d_hint(sb + 128 * 128, ts, xs, y, fb, pol);
      }
      cursor_next_unit(c);
    }
    ++it;
    ++c.k;
    *reinterpret_cast<volatile unsigned*>(&sh.issued) = it;
  }
  // never leave with copies in flight: the last uses issued (whether or not
  // the consumers took them) have landed before the producer returns, all
  // within one bounded wait
  const unsigned long long deadline = dev::globaltimer_ns() + kWaitLimitNs;
  for (unsigned u = it > (unsigned)kStages ? it - kStages : 0u; u < it; ++u)
    dev::mbar_wait_until(dev::smem_u32(&sh.full[u % kStages]), (u / kStages) & 1, deadline);
}

// ============================================================== the L2 prefetch
// Lane 0 of the prefetch warp walks the same schedule kPfAhead uses ahead of
// the producer and pulls each use's boxes toward L2.  A wait for a step's
// inputs then does not stop the HBM stream: the ring's copies after it read
// L2.  (Key blocks that hold this call's rows are not written yet and are
// skipped.)  It runs in a warp of its own: a lane sharing the producer's warp
// would sleep while the producer sleeps on a stage.
__device__ __noinline__ void prefetcher(const PassParams& p) {
  Cursor c;
  c.l = 0;
  c.ph = 0;
  cursor_enter(p, c);
  unsigned it = 0;
  for (;;) {
    if (c.k >= c.n) {
      if (++c.ph == kPassPhases) {
        c.ph = 0;
        if (++c.l == p.L) return;
      }
      cursor_enter(p, c);
      continue;
    }
    // stay kPfAhead uses ahead of the copies, no further (L2 holds the window)
    if (it >= *reinterpret_cast<volatile unsigned*>(&sh.issued) + kPfAhead) {
      const unsigned long long t0 = dev::globaltimer_ns();
      while (it >= *reinterpret_cast<volatile unsigned*>(&sh.issued) + kPfAhead) {
        if (*reinterpret_cast<volatile int*>(&sh.abort) || dev::globaltimer_ns() - t0 > kWaitLimitNs) return;
        __nanosleep(100);
      }
    }
    if (c.ph == kPhAttn) {
      if ((c.b + 1) * kAttnKeys <= p.rows.P) {
        if ((c.k & 1) == 0) {
          dev::tma_prefetch_2d(&p.tkv, 0, c.kb + c.b * kAttnKeys);
          dev::tma_prefetch_2d(&p.tkv, 64, c.kb + c.b * kAttnKeys);
        } else {
          dev::tma_prefetch_2d(&p.tvt, c.b * kAttnKeys, c.vb);
        }
      }
      if (c.k & 1) ++c.b;
    } else {
      const CUtensorMap* tw = &c.Ly->tw[c.wi];
      const CUtensorMap* ts = &c.Ly->ts[c.wi];
      const int x = c.ks * 128, xs = c.ks * 8, y = c.row0;
      dev::tma_prefetch_2d(tw, x, y);
      dev::tma_prefetch_2d(ts, xs, y);
      if (c.pair) {
        dev::tma_prefetch_2d(tw + 1, x, y);
        dev::tma_prefetch_2d(ts + 1, xs, y);
      }
      cursor_next_unit(c);
    }
    ++it;
    ++c.k;
  }
}

// ============================================================== consumers
struct Cons {
  const PassParams& p;
  uint32_t ring;
  uint8_t* work;        // generic pointer to the work area
  uint32_t work_s;      // its shared address
  unsigned it;          // ring uses taken so far (the producer issues them in the same order)
  int tid, warp, lane;
  bool ok;              // uniform after each cons_sync

  __device__ __forceinline__ Cons(const PassParams& pp, uint32_t r, uint8_t* w, uint32_t ws)
      : p(pp), ring(r), work(w), work_s(ws), it(0) {
    tid = threadIdx.x;
    warp = tid >> 5;
    lane = tid & 31;
    ok = true;
  }

  __device__ __forceinline__ volatile int& abort_flag() { return *reinterpret_cast<volatile int*>(&sh.abort); }

  // one thread waits for a counter; everyone learns the outcome at the barrier
  __device__ __forceinline__ bool wait_dep(int idx, int count) {
    if (tid == 0 && !abort_flag()) {
      const int* ctr = p.done + idx;
      const int target = (int)p.epoch * count;
      const unsigned long long t0 = dev::globaltimer_ns();
      for (unsigned n = 0;; ++n) {
        if (ld_acquire(ctr) - target >= 0) break;
        __nanosleep(kCountBackoffNs);
        if ((n & 15u) == 15u && dev::status_set(p.status)) {
          abort_flag() = 1;
          break;
        }
        if (dev::globaltimer_ns() - t0 > kWaitLimitNs) {
          give_up(p.status, p.diag, kSiteConsCount, idx, ld_acquire(ctr));
          abort_flag() = 1;
          break;
        }
      }
    }
    ok = !cons_sync_any(abort_flag() != 0);
    return ok;
  }

  // wait for ring use u (its stage full) and return the stage's shared
  // address; a failed wait marks the CTA aborted (every warp still passes
  // every use, so the ring's phases stay in step)
  __device__ __forceinline__ uint32_t wait_use(unsigned u, bool& good) {
    const int st = (int)(u % kStages);
    const uint32_t bar = dev::smem_u32(&sh.full[st]);
    const uint32_t parity = (u / kStages) & 1;
    bool got = false;
    if (!abort_flag()) got = ring_wait(bar, parity, p.status, p.diag, kSiteConsRing, (int)u);
    good = __all_sync(0xffffffffu, got);
    if (!good && lane == 0) abort_flag() = 1;
    return ring + st * kStage;
  }
  __device__ __forceinline__ void release_use(unsigned u) {
    __syncwarp();
    if (lane == 0) dev::mbar_arrive(dev::smem_u32(&sh.empty[u % kStages]));
  }

  // ---------------------------------------------------------- activations
  // x for the unit at k-step ks: rows [0, m) of 256 inputs, bf16, in the
  // GEMV's swizzled box layout; a warp stages rows warp and warp + 8, a lane
  // one 8-input chunk of each
  struct Chunk {
    float4 h0, h1;
    uint4 g;
  };
  __device__ __forceinline__ void chunk_load(int ph, const __nv_bfloat16* gain, int ks, int n, Chunk& c) const {
    const int k = ks * kGemvKStep + 8 * lane;
    if (ph == kPhQKV || ph == kPhGU) {
      const float4* hp = reinterpret_cast<const float4*>(p.h + (long long)n * p.H + k);
      c.h0 = __ldcg(hp);
      c.h1 = __ldcg(hp + 1);
      c.g = *reinterpret_cast<const uint4*>(gain + k);
    } else {
      const __nv_bfloat16* src = ph == kPhO ? p.o + (long long)n * p.Hq * p.d : p.z + (long long)n * p.F;
      c.g = __ldcg(reinterpret_cast<const uint4*>(src + k));
    }
  }
  template <int NT>
  __device__ __forceinline__ void chunk_store(int ph, const Chunk& c, int n, uint32_t xbuf) const {
    const int k8 = lane;
    uint4 v = c.g;
    if (ph == kPhQKV || ph == kPhGU) {
      const float r = sh.rscale[n];
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&c.g);
      const float2 g0 = __bfloat1622float2(g2[0]), g1 = __bfloat1622float2(g2[1]);
      const float2 g2f = __bfloat1622float2(g2[2]), g3 = __bfloat1622float2(g2[3]);
      v.x = dev::pack_bf16x2(c.h0.x * r * g0.x, c.h0.y * r * g0.y);
      v.y = dev::pack_bf16x2(c.h0.z * r * g1.x, c.h0.w * r * g1.y);
      v.z = dev::pack_bf16x2(c.h1.x * r * g2f.x, c.h1.y * r * g2f.y);
      v.w = dev::pack_bf16x2(c.h1.z * r * g3.x, c.h1.w * r * g3.y);
    }
    const uint32_t addr = xbuf + (k8 >> 3) * (NT * 1024) + dev::swz128((uint32_t)n, (uint32_t)(k8 & 7));
    // no memory clobber: the next items' global loads may be issued before
    // this store; the barrier after the staging orders it before the reads
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w));
  }

  // RMSNorm factors of the call's rows from the per-tile sums (fixed order)
  __device__ __forceinline__ void row_scales() {
    for (int n = warp; n < p.m; n += kWarps) {
      float v = 0.f;
      for (int j = lane; j < p.nss; j += 32) v += __ldcg(p.ss + (long long)n * p.nss + j);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) sh.rscale[n] = rsqrtf(v / p.H + p.eps);
    }
  }

  // stage x of nslot units from unit ua on (slot i: unit ua + i): a warp per
  // (unit, row), a lane per 8 inputs.  O and DOWN copy bf16 rows of o and z
  // with asynchronous copies, all in flight at once; QKV and GU convert
  // RMSNorm(h) * g two items at a time (both items' loads in flight before
  // the first store).  Rows from m to 8 * NT are left as they are: they feed
  // output columns that are never stored.
  template <int NT>
  __device__ __forceinline__ void stage(int ph, const __nv_bfloat16* gain, int ua, int nslot, int ksteps) {
    constexpr int kUnitX = 4 * NT * 1024;
    const int items = nslot * p.m;
    if (ph == kPhO || ph == kPhDown) {
      for (int sn = warp; sn < items; sn += kWarps) {
        const int slot = sn / p.m, n = sn - slot * p.m;
        const int k = ((ua + slot) % ksteps) * kGemvKStep + 8 * lane;
        const __nv_bfloat16* src = ph == kPhO ? p.o + (long long)n * p.Hq * p.d : p.z + (long long)n * p.F;
        const uint32_t dst = work_s + slot * kUnitX + (lane >> 3) * (NT * 1024) + dev::swz128((uint32_t)n, (uint32_t)(lane & 7));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + k) : "memory");
      }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
      return;
    }
    for (int sn = warp; sn < items; sn += 2 * kWarps) {
      Chunk c0, c1;
      const int sn1 = sn + kWarps;
      const int slot0 = sn / p.m, n0 = sn - slot0 * p.m;
      const int slot1 = sn1 / p.m, n1 = sn1 - slot1 * p.m;
      chunk_load(ph, gain, (ua + slot0) % ksteps, n0, c0);
      if (sn1 < items) chunk_load(ph, gain, (ua + slot1) % ksteps, n1, c1);
      chunk_store<NT>(ph, c0, n0, work_s + slot0 * kUnitX);
      if (sn1 < items) chunk_store<NT>(ph, c1, n1, work_s + slot1 * kUnitX);
    }
  }

  // ---------------------------------------------------------- one projection step
  template <int NT>
  __device__ __forceinline__ void projection(int l, int ph) {
    const Proj j = proj_of(p, ph);
    const int units = j.tiles * j.ksteps;
    int u0, u1;
    unit_range(units, p.ctas, blockIdx.x, u0, u1);
    const int nk = u1 - u0;
    if (nk <= 0) return;
    const PassLayer* Ly = p.layers + l;
    // inputs: the previous step of this layer, or the previous layer's down step
    const int dep = ph == kPhQKV ? (l == 0 ? p.L * kPassPhases : done_index(l - 1, kPhDown))
                                 : done_index(l, ph - 1);
    if (!wait_dep(dep, l == 0 && ph == kPhQKV ? p.nss : done_count(p, ph == kPhQKV ? kPhDown : ph - 1)))
      return;
    const bool norm = ph == kPhQKV || ph == kPhGU;
    const __nv_bfloat16* gain = ph == kPhQKV ? Ly->norm_attn : Ly->norm_ffn;
    if (norm) {
      row_scales();
      cons_sync();
    }
    float* ct = reinterpret_cast<float*>(work);   // the epilogue's tile buffer (after the units)
    constexpr int kUnitX = 4 * NT * 1024;          // staged activations of one unit
    constexpr int kChunk = kXArea / kUnitX;        // units staged at a time (16 or 8)
    // warp role: 16 weight rows of the tile, all 256 inputs of a unit
    const int r = lane >> 2, c = lane & 3;
    const int rho0 = warp * 16 + r;
    float acc[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[t][e] = 0.f;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    // a unit's activations depend on its k-step alone: when the step has at
    // most kChunk k-steps, each is staged once and the units that repeat it
    // reuse its slot; otherwise the units go kChunk at a time
    const bool once = j.ksteps <= kChunk;
    const int span = once ? nk : kChunk;
    for (int c0 = 0; c0 < nk; c0 += span) {
      const int cn = min(span, nk - c0);
      const int nslot = once ? min(nk, j.ksteps) : cn;
      if (c0 > 0) cons_sync();   // the previous chunk's activations are read
      stage<NT>(ph, gain, u0 + c0, nslot, j.ksteps);
      cons_sync();
      // running (tile, k-step) of the unit and its activation slot
      int ks_c = (u0 + c0) % j.ksteps, tile_c = (u0 + c0) / j.ksteps, slot = 0;
      for (int i = c0; i < c0 + cn; ++i) {
        const uint32_t xb = work_s + slot * kUnitX;
        bool good;
        const uint32_t wt = wait_use(it, good);
        if (good) {
          const uint32_t stile = wt + 128 * 128;
          const uint4 sc0 = dev::lds128(stile + rho0 * 16);
          const uint4 sc1 = dev::lds128(stile + (rho0 + 8) * 16);
          const __half* s0h = reinterpret_cast<const __half*>(&sc0);
          const __half* s1h = reinterpret_cast<const __half*>(&sc1);
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint32_t w0 = dev::lds32(wt + dev::swz128(rho0, g) + 4 * c);
            const uint32_t w1 = dev::lds32(wt + dev::swz128(rho0 + 8, g) + 4 * c);
            uint32_t q0[4], q1[4];
            codes_bf16(w0, q0);
            codes_bf16(w1, q1);
            const uint32_t a_lo[4] = {q0[0], q1[0], q0[1], q1[1]};
            const uint32_t a_hi[4] = {q0[2], q1[2], q0[3], q1[3]};
            const float sr0 = __half2float(s0h[g]);
            const float sr1 = __half2float(s1h[g]);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const int n = t * 8 + (lane & 7);
              const int q = lane >> 3;
              uint32_t b0, b1, b2, b3;
              dev::ldmatrix_x4(xb + (g >> 1) * (NT * 1024) + dev::swz128(n, 4 * (g & 1) + q), b0, b1, b2, b3);
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
        release_use(it);
        ++it;
        // the tile's partial of this CTA: each warp stores its 16 rows
        if (ks_c == j.ksteps - 1 || i == nk - 1) {
          const int tile = tile_c;
          const int first = owner_of((long long)tile * j.ksteps, units, p.ctas);
          float* tp = p.part + ((long long)tile * p.maxc[ph] + (blockIdx.x - first)) * (kGemvMaxCols * kGemvRows);
#pragma unroll
          for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int tok = t * 8 + 2 * c + (e & 1);
              const int row = rho0 + (e >> 1) * 8;
              if (tok < p.m) tp[tok * kGemvRows + row] = acc[t][e];
              acc[t][e] = 0.f;
            }
        }
        if (++ks_c == j.ksteps) {
          ks_c = 0;
          ++tile_c;
        }
        if (++slot == j.ksteps && once) slot = 0;
      }
    }
    // one arrival per tile this CTA touched; the last arrival owns the epilogue
    if (tid == 0) sh.n_own = 0;
    ok = !cons_sync_any(abort_flag() != 0);
    if (!ok) return;
    {
      const int t_first = u0 / j.ksteps, t_last = (u1 - 1) / j.ksteps;
      const int tile = t_first + tid;
      if (tile <= t_last) {
        const long long tu0 = (long long)tile * j.ksteps;
        const int ncon = owner_of(tu0 + j.ksteps - 1, units, p.ctas) - owner_of(tu0, units, p.ctas) + 1;
        const int done = dev::atom_add_acq_rel(p.tile_cnt + tile, 1) + 1;
        if (done == ncon) {
          p.tile_cnt[tile] = 0;   // ready for the next use
          const int k = atomicAdd(&sh.n_own, 1);
          if (k < kMaxOwn) sh.own[k] = tile;
        }
      }
    }
    cons_sync();
    const int n_done = min(sh.n_own, kMaxOwn);
    for (int k = 0; k < n_done; ++k) {
      const int tile = sh.own[k];
      epilogue(l, ph, j, units, tile, ct);
      cons_sync();
      if (tid == 0) red_release_add(p.done + done_index(l, ph), 1);
    }
  }

  // add a tile's partials in contributor order, then the step's epilogue
  __device__ __forceinline__ void epilogue(int l, int ph, const Proj& j, int units, int tile, float* ct) {
    const long long tu0 = (long long)tile * j.ksteps;
    const int first = owner_of(tu0, units, p.ctas);
    const int ncon = owner_of(tu0 + j.ksteps - 1, units, p.ctas) - first + 1;
    const int s = seg_of(j, tile);
    const int row0 = row0_of(j, tile, s);
    const bool resid = ph == kPhO || ph == kPhDown;
    const int nv_h = resid ? min(kGemvRows, p.H - row0) : 0;
    const float* t0p = p.part + (long long)tile * p.maxc[ph] * (kGemvMaxCols * kGemvRows);
    const bool last_layer = l == p.L - 1;
    for (int idx = tid; idx < p.m * (kGemvRows / 4); idx += kCons) {
      const int tok = idx / (kGemvRows / 4), r4 = (idx % (kGemvRows / 4)) * 4;
      const float* src = t0p + tok * kGemvRows + r4;
      float4 hv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (resid && r4 < nv_h) hv = __ldcg(reinterpret_cast<const float4*>(p.h + (long long)tok * p.H + row0 + r4));
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = 0; j0 < ncon; j0 += 4) {
        float4 w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (j0 + q < ncon) w[q] = __ldcg(reinterpret_cast<const float4*>(src + (long long)(j0 + q) * (kGemvMaxCols * kGemvRows)));
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (j0 + q < ncon) {
            v.x += w[q].x; v.y += w[q].y; v.z += w[q].z; v.w += w[q].w;
          }
      }
      if (resid) {
        // h += y, the new rows' sum of squares over this 128-column tile (one
        // warp per row, fixed order), and the bf16 output on the last layer
        float ssq = 0.f;
        if (r4 < nv_h) {
          hv.x += v.x; hv.y += v.y; hv.z += v.z; hv.w += v.w;
          *reinterpret_cast<float4*>(p.h + (long long)tok * p.H + row0 + r4) = hv;
          if (ph == kPhDown && p.trace)
            *reinterpret_cast<float4*>(p.trace + ((long long)(l + 1) * p.trace_rows + tok) * p.H + row0 + r4) = hv;
          ssq = hv.x * hv.x + hv.y * hv.y + hv.z * hv.z + hv.w * hv.w;
          if (ph == kPhDown && last_layer && p.out) {
            uint2 o;
            o.x = dev::pack_bf16x2(hv.x, hv.y);
            o.y = dev::pack_bf16x2(hv.z, hv.w);
            *reinterpret_cast<uint2*>(p.out + (long long)tok * p.H + row0 + r4) = o;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
        if (lane == 0) p.ss[(long long)tok * p.nss + row0 / kGemvRows] = ssq;
      } else {
        *reinterpret_cast<float4*>(ct + tok * kCtLd + r4) = v;
      }
    }
    if (resid) return;
    cons_sync();
    if (ph == kPhGU) {
      const int nv = min(64, p.F - row0);
      for (int idx = tid; idx < p.m * 64; idx += kCons) {
        const int tok = idx >> 6, jj = idx & 63;
        if (jj >= nv) continue;
        const float g = ct[tok * kCtLd + jj], u = ct[tok * kCtLd + 64 + jj];
        const float sg = g / (1.f + expf(-g));
        p.z[(long long)tok * p.F + row0 + jj] = __float2bfloat16_rn(sg * u);
      }
      return;
    }
    // QKV: a tile is one head (d = 128) or two (d = 64) of q, k or v
    const int d = p.d, half = d >> 1;
    const int nv = min(kGemvRows, rows_of(j, s) - row0);
    const int hd0 = row0 / d;
    const long long koff = (long long)(2 * l) * p.Hkv * p.cap * d;
    const long long voff = (long long)(2 * l + 1) * p.Hkv * p.cap * d;
    if (s < 2) {
      const int npairs = nv >> 1;
      for (int idx = tid; idx < p.m * npairs; idx += kCons) {
        const int t = idx / npairs, pr = idx % npairs;
        const int hh = pr / half, jj = pr % half;
        const int col = hh * d + jj;
        const float x1 = ct[t * kCtLd + col];
        const float x2 = ct[t * kCtLd + col + half];
        const float2 cs = p.rope[(long long)t * half + jj];
        const float y1 = x1 * cs.x - x2 * cs.y;
        const float y2 = x2 * cs.x + x1 * cs.y;
        const int hd = hd0 + hh;
        __nv_bfloat16* dst =
            s == 0 ? p.q + q_row(p.rows, t, hd / p.G, hd % p.G, p.G, p.Hq) * d
                   : kv_base() + koff + ((long long)hd * p.cap + row_store(p.rows, t)) * d;
        dst[jj] = __float2bfloat16_rn(y1);
        dst[jj + half] = __float2bfloat16_rn(y2);
      }
    } else {
      for (int idx = tid; idx < p.m * nv; idx += kCons) {
        const int t = idx % p.m, col = idx / p.m;
        const int hd = hd0 + col / d, e = col % d;
        kv_base()[voff + ((long long)hd * d + e) * p.cap + row_store(p.rows, t)] =
            __float2bfloat16_rn(ct[t * kCtLd + col]);
      }
    }
  }

  // the slot's K/V region (layer 0, K) as bf16 elements
  __device__ __forceinline__ __nv_bfloat16* kv_base() const { return p.arena + p.kv_slot; }

  // ---------------------------------------------------------- the embedding
  // h = float(hidden) and the per-tile sums of squares: item t (one per
  // 128-column tile, whatever the row count, so the counter's count per call
  // is fixed) covers tile t of every row, on warp 0 of a CTA
  __device__ void embed() {
    if (warp != 0) return;
    for (int t = blockIdx.x; t < p.nss; t += p.ctas) {
      const int k = t * kGemvRows + 4 * lane;
      for (int i = 0; i < p.m; ++i) {
        float ssq = 0.f;
        if (k < p.H) {
          const uint2 raw = *reinterpret_cast<const uint2*>(p.hidden + (long long)i * p.H + k);
          const float2 x01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
          const float2 x23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
          const float4 x = make_float4(x01.x, x01.y, x23.x, x23.y);
          *reinterpret_cast<float4*>(p.h + (long long)i * p.H + k) = x;
          if (p.trace) *reinterpret_cast<float4*>(p.trace + (long long)i * p.H + k) = x;
          ssq = x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
        if (lane == 0) p.ss[(long long)i * p.nss + t] = ssq;
      }
      __syncwarp();
      if (lane == 0) red_release_add(p.done + p.L * kPassPhases, 1);
    }
  }

  // ---------------------------------------------------------- split merge
  // The last split of a KV head to finish merges every split's partial (O,
  // max, sum) of the head's R rows into o, in split order.  First the weights
  // 2^(m_s - M) and 1 / sum_s w_s l_s of every row (a warp per row, a lane per
  // split, the rows of a warp's loads in flight together), into shared memory;
  // then rows in chunks that fit the work area: every (row, split) partial of
  // the chunk copied in with asynchronous copies, all in flight at once, and a
  // thread per (row, four head dims) adds them up.
  __device__ __forceinline__ void merge(int kv, int R) {
    constexpr int D = kAttnD;
    const int ns = p.nsplit;
    const long long stride = (long long)kPassMaxAttnRows;   // rows per split partial
    float* wsm = reinterpret_cast<float*>(work);            // [R][ns] weights
    float* inv = wsm + kPassMaxAttnRows * kMaxSplits;       // [R] 1 / denominator
    const uint32_t stage_s = work_s + (kPassMaxAttnRows * kMaxSplits + kPassMaxAttnRows) * 4;
    const float* stage = reinterpret_cast<const float*>(work + (stage_s - work_s));
    constexpr int kStageBytes = kWork - (kPassMaxAttnRows * kMaxSplits + kPassMaxAttnRows) * 4;
    const float2* mlk = p.ml + (long long)kv * ns * stride;
    constexpr int kRowsW = kPassMaxAttnRows / kWarps;        // rows of one warp (at most)
    float2 a[kRowsW], b[kRowsW];
#pragma unroll
    for (int q = 0; q < kRowsW; ++q) {
      const int row = warp + q * kWarps;
      a[q] = row < R && lane < ns ? __ldcg(mlk + lane * stride + row) : make_float2(-INFINITY, 0.f);
      b[q] = row < R && lane + 32 < ns ? __ldcg(mlk + (lane + 32) * stride + row) : make_float2(-INFINITY, 0.f);
    }
#pragma unroll
    for (int q = 0; q < kRowsW; ++q) {
      const int row = warp + q * kWarps;
      if (row >= R) continue;
      float M = fmaxf(a[q].x, b[q].x);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
      const float w0 = a[q].x == -INFINITY ? 0.f : exp2f(a[q].x - M);
      const float w1 = b[q].x == -INFINITY ? 0.f : exp2f(b[q].x - M);
      float den = w0 * a[q].y + w1 * b[q].y;
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o2);
      if (lane < ns) wsm[row * ns + lane] = w0;
      if (lane + 32 < ns) wsm[row * ns + lane + 32] = w1;
      if (lane == 0) inv[row] = 1.f / den;
    }
    const int rows_chunk = max(1, min(R, kStageBytes / (ns * D * 4)));
    for (int r0 = 0; r0 < R; r0 += rows_chunk) {
      const int rc = min(rows_chunk, R - r0);
      cons_sync();   // weights written; the previous chunk's partials read
      // (row, split, 16-byte piece): 32 pieces per 512-byte partial row
      for (int idx = tid; idx < rc * ns * (D / 4); idx += kCons) {
        const int pc = idx % (D / 4), rs = idx / (D / 4);
        const int sp = rs % ns, row = r0 + rs / ns;
        const float* src = p.opart + (((long long)kv * ns + sp) * stride + row) * D + 4 * pc;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(stage_s + 16u * (uint32_t)idx), "l"(src)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
      cons_sync();
      for (int idx = tid; idx < rc * (D / 4); idx += kCons) {
        const int pc = idx % (D / 4), rr = idx / (D / 4), row = r0 + rr;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int sp = 0; sp < ns; ++sp) {
          const float w = wsm[row * ns + sp];
          const float4 x = reinterpret_cast<const float4*>(stage)[(rr * ns + sp) * (D / 4) + pc];
          acc.x += w * x.x; acc.y += w * x.y; acc.z += w * x.z; acc.w += w * x.w;
        }
        const float iv = inv[row];
        const int tok = row / p.G, head = kv * p.G + row % p.G;
        uint2 v;
        v.x = dev::pack_bf16x2(acc.x * iv, acc.y * iv);
        v.y = dev::pack_bf16x2(acc.z * iv, acc.w * iv);
        *reinterpret_cast<uint2*>(p.o + (long long)tok * p.Hq * D + head * D + 4 * pc) = v;
      }
    }
  }

  // ---------------------------------------------------------- attention
  __device__ __forceinline__ void attention(int l) {
    const Item item = item_of(p, blockIdx.x);
    if (!item.any) return;
    if (!wait_dep(done_index(l, kPhQKV), done_count(p, kPhQKV))) return;
    const int D = kAttnD;
    const int R = p.G * p.m;
    const int RT = (R + 15) / 16;
    const int KW = RT == 1 ? 4 : (RT == 2 ? 2 : 1);
    const int nw = RT * KW;   // warp pairs
    const int kv = item.kv;
    // this KV head's query rows (row = token * G + head in group), zero-padded
    // to whole 16-row tiles, in shared memory
    __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(work + (KW > 1 ? kMergeBytes : 0));
    const __nv_bfloat16* qsrc = p.q + (long long)kv * p.m * p.G * D;   // [m][G][D] of this KV head
    for (int idx = tid; idx < RT * 16 * (D / 8); idx += kCons) {
      const int row = idx / (D / 8), c8 = idx % (D / 8);
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (row < R) v = __ldcg(reinterpret_cast<const uint4*>(qsrc + (long long)row * D) + c8);
      reinterpret_cast<uint4*>(qs + row * D)[c8] = v;
    }
    cons_sync();
    // warps: (row tile, key-parallel lane kw, half of the head dims dh); both
    // halves of a pair form the same scores and softmax, each accumulates
    // its 64 output dims
    const int aw = warp < 2 * nw ? warp : -1;
    const int dh = aw >= 0 ? (aw & 1) : 0;
    const int pw = aw >= 0 ? (aw >> 1) : 0;
    const int rt = pw / KW, kw = pw % KW;
    const int r = lane >> 2, c = lane & 3;
    const int rho[2] = {rt * 16 + r, rt * 16 + r + 8};
    int vis_lo[2], vis_hi[2];
    bool real[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      real[h] = rho[h] < R;
      const int tok = real[h] ? rho[h] / p.G : 0;
      const int b = row_branch(p.rows, tok);
      vis_lo[h] = p.rows.P + p.rows.off[b];
      vis_hi[h] = real[h] ? p.rows.P + tok : -1;
    }
    constexpr int DH = D / 2;
    float o[DH / 8][4];
#pragma unroll
    for (int i = 0; i < DH / 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    const int P = p.rows.P;
    for (int b = item.b0; b < item.b1; ++b) {
      bool gk, gv;
      const uint32_t kt = wait_use(it, gk);
      const uint32_t vt = wait_use(it + 1, gv);
      if (aw >= 0 && gk && gv && (b - item.b0) % KW == kw) {
        // the block's 64 keys in two halves of 32: S = Q K^T, mask (the prefix
        // and the row's own branch up to itself), online softmax in log2
        // units, then O += P V for this warp's 64 head dims
#pragma unroll 1
        for (int hf = 0; hf < 2; ++hf) {
          const int key0 = b * kAttnKeys + 32 * hf;
          float s[4][4];
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[nt][e] = 0.f;
#pragma unroll 2
          for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t qa[4];
            const __nv_bfloat16* q0 = qs + rho[0] * D + kk * 16 + 2 * c;
            const __nv_bfloat16* q1 = qs + rho[1] * D + kk * 16 + 2 * c;
            qa[0] = *reinterpret_cast<const uint32_t*>(q0);
            qa[1] = *reinterpret_cast<const uint32_t*>(q1);
            qa[2] = *reinterpret_cast<const uint32_t*>(q0 + 8);
            qa[3] = *reinterpret_cast<const uint32_t*>(q1 + 8);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
              const int q = lane >> 3;
              const int key = 32 * hf + 8 * (2 * np + (q >> 1)) + (lane & 7);
              const int chunk = 2 * kk + (q & 1);
              uint32_t b0r, b1r, b2r, b3r;
              dev::ldmatrix_x4(kt + (chunk >> 3) * (kAttnKeys * 128) + dev::swz128(key, chunk & 7), b0r, b1r,
                               b2r, b3r);
              dev::mma_bf16_16816(s[2 * np], qa, b0r, b1r, s[2 * np]);
              dev::mma_bf16_16816(s[2 * np + 1], qa, b2r, b3r, s[2 * np + 1]);
            }
          }
          float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int jk = key0 + 8 * nt + 2 * c + (e & 1);
              const int h = e >> 1;
              const bool vis = real[h] && (jk < P || (jk >= vis_lo[h] && jk <= vis_hi[h]));
              const float v = vis ? s[nt][e] * p.scale_log2 : -INFINITY;
              s[nt][e] = v;
              mx[h] = fmaxf(mx[h], v);
            }
          float corr[2], muse[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
            mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
            const float mnew = fmaxf(mrow[h], mx[h]);
            muse[h] = mnew == -INFINITY ? 0.f : mnew;
            corr[h] = exp2f(mrow[h] - muse[h]);
            mrow[h] = mnew;
            lrow[h] *= corr[h];
          }
#pragma unroll
          for (int i = 0; i < DH / 8; ++i) {
            o[i][0] *= corr[0]; o[i][1] *= corr[0];
            o[i][2] *= corr[1]; o[i][3] *= corr[1];
          }
#pragma unroll
          for (int nt = 0; nt < 4; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float pv = exp2f(s[nt][e] - muse[e >> 1]);
              s[nt][e] = pv;
              lrow[e >> 1] += pv;
            }
          // P as the A operand (16 keys a step); V^T rows are head elements
#pragma unroll 1
          for (int ks = 0; ks < 2; ++ks) {
            uint32_t pa[4];
            pa[0] = dev::pack_bf16x2(s[2 * ks][0], s[2 * ks][1]);
            pa[1] = dev::pack_bf16x2(s[2 * ks][2], s[2 * ks][3]);
            pa[2] = dev::pack_bf16x2(s[2 * ks + 1][0], s[2 * ks + 1][1]);
            pa[3] = dev::pack_bf16x2(s[2 * ks + 1][2], s[2 * ks + 1][3]);
#pragma unroll
            for (int dp = 0; dp < DH / 16; ++dp) {
              const int q = lane >> 3;
              const int drow = dh * DH + 16 * dp + 8 * (q >> 1) + (lane & 7);
              const int chunk = 4 * hf + 2 * ks + (q & 1);
              uint32_t b0r, b1r, b2r, b3r;
              dev::ldmatrix_x4(vt + dev::swz128(drow, chunk), b0r, b1r, b2r, b3r);
              dev::mma_bf16_16816(o[2 * dp], pa, b0r, b1r, o[2 * dp]);
              dev::mma_bf16_16816(o[2 * dp + 1], pa, b2r, b3r, o[2 * dp + 1]);
            }
          }
        }
      }
      release_use(it);
      release_use(it + 1);
      it += 2;
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 1);
      lrow[h] += __shfl_xor_sync(0xffffffffu, lrow[h], 2);
    }
    const long long pbase = (long long)(kv * p.nsplit + item.split) * kPassMaxAttnRows;
    if (KW > 1) {
      // the KW warps of a (row tile, dims half) merge their states through
      // shared memory
      float* mb = reinterpret_cast<float*>(work);
      if (aw >= 0) {
        float* mine = mb + aw * kMergeState;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = r + 8 * h;
#pragma unroll
          for (int i = 0; i < DH / 8; ++i)
            *reinterpret_cast<float2*>(mine + row * DH + 8 * i + 2 * c) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
          if (c == 0) {
            mine[16 * DH + row] = mrow[h];
            mine[16 * DH + 16 + row] = lrow[h];
          }
        }
      }
      cons_sync();
      if (aw >= 0 && kw == 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int row = r + 8 * h;
          float M = -INFINITY;
          float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (w < KW) M = fmaxf(M, mb[(aw + 2 * w) * kMergeState + 16 * DH + row]);
          float L = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w)
            if (w < KW) {
              const float mw = mb[(aw + 2 * w) * kMergeState + 16 * DH + row];
              sc[w] = mw == -INFINITY ? 0.f : exp2f(mw - M);
              L += sc[w] * mb[(aw + 2 * w) * kMergeState + 16 * DH + 16 + row];
            }
#pragma unroll
          for (int i = 0; i < DH / 8; ++i) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int w = 0; w < 4; ++w)
              if (w < KW) {
                const float2 x = *reinterpret_cast<const float2*>(mb + (aw + 2 * w) * kMergeState + row * DH + 8 * i + 2 * c);
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
    }
    // this split's partial (unnormalised O, max, sum) of every real row
    if (aw >= 0 && kw == 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (!real[h]) continue;
        float* dst = p.opart + (pbase + rho[h]) * D + dh * DH;
#pragma unroll
        for (int i = 0; i < DH / 8; ++i)
          *reinterpret_cast<float2*>(dst + 8 * i + 2 * c) = make_float2(o[i][2 * h], o[i][2 * h + 1]);
        if (c == 0 && dh == 0) p.ml[pbase + rho[h]] = make_float2(mrow[h], lrow[h]);
      }
    }
    cons_sync();
    if (tid == 0) {
      const int n = dev::atom_add_acq_rel(p.head_cnt + kv, 1) + 1;
      sh.merge_last = n == p.nsplit;
      if (n == p.nsplit) p.head_cnt[kv] = 0;
    }
    cons_sync();
    if (!sh.merge_last) return;
    // the last split merges every split's rows in split order into o
    merge(kv, R);
    cons_sync();
    if (tid == 0) red_release_add(p.done + done_index(l, kPhAttn), 1);
  }

  // ---------------------------------------------------------- the output head's norm
  __device__ void head_norm() {
    if (!p.head_gain || (int)blockIdx.x >= p.m) return;
    if (!wait_dep(done_index(p.L - 1, kPhDown), done_count(p, kPhDown))) return;
    const int i = blockIdx.x;
    if (warp == 0) {
      float v = 0.f;
      for (int j = lane; j < p.nss; j += 32) v += __ldcg(p.ss + (long long)i * p.nss + j);
#pragma unroll
      for (int o2 = 16; o2 > 0; o2 >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o2);
      if (lane == 0) sh.rscale[0] = rsqrtf(v / p.H + p.eps);
    }
    cons_sync();
    const float rs = sh.rscale[0];
    for (int k = tid; k < p.H; k += kCons)
      p.a_head[(long long)i * p.H + k] =
          __float2bfloat16_rn(__ldcg(p.h + (long long)i * p.H + k) * rs * __bfloat162float(p.head_gain[k]));
  }
};

template <int NT>
__global__ void __launch_bounds__(kThreads, 1) pass_kernel(const __grid_constant__ PassParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t ring = base;
  const uint32_t work_s = base + kStages * kStage;
  uint8_t* work = smem_raw + (work_s - raw);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      dev::mbar_init(dev::smem_u32(&sh.full[i]), 1);
      dev::mbar_init(dev::smem_u32(&sh.empty[i]), kWarps);
    }
    // a wait has given up earlier: leave before any copy
    sh.abort = dev::status_set(p.status) ? 1 : 0;
    sh.n_own = 0;
    sh.merge_last = 0;
    sh.issued = 0;
    sh.item = item_of(p, blockIdx.x);
    for (int ph = 0; ph < kPassPhases; ++ph) {
      sh.u0[ph] = sh.u1[ph] = 0;
      if (ph == kPhAttn) continue;
      const Proj j = proj_of(p, ph);
      unit_range(j.tiles * j.ksteps, p.ctas, blockIdx.x, sh.u0[ph], sh.u1[ph]);
    }
    dev::fence_mbar_init();
  }
  __syncthreads();
  if (sh.abort) return;
  if (threadIdx.x >= kCons) {
    // the producer and prefetch warps: one lane each, the others have no work
    if (threadIdx.x == kCons) producer(p, ring);
    if (threadIdx.x == kCons + 32) prefetcher(p);
    return;
  }
  Cons cs(p, ring, work, work_s);
  cs.embed();
  for (int l = 0; l < p.L && cs.ok; ++l) {
#pragma unroll 1
    for (int ph = 0; ph < kPassPhases && cs.ok; ++ph) {
      if (ph == kPhAttn) cs.attention(l);
      else cs.template projection<NT>(l, ph);
    }
  }
  if (cs.ok) cs.head_norm();
  // a consumer that stops early tells the producer, which then stops issuing
  if (!cs.ok && threadIdx.x == 0) *reinterpret_cast<volatile int*>(&sh.abort) = 1;
}

int g_ctas = 0;

}  // namespace

int pass_ctas() { return g_ctas; }

cudaError_t pass_setup() {
  cudaError_t e = cudaFuncSetAttribute(pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  int dev = 0, sms = 0, per = 0;
  if (e == cudaSuccess) e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, pass_kernel<2>, kThreads, kSmem);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(pass_kernel<1>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess) e = cudaFuncSetAttribute(pass_kernel<2>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
  if (e == cudaSuccess) g_ctas = per >= 1 ? sms : 0;
  return e;
}

cudaError_t launch_pass(const PassParams& p, int nt, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = st;
  // every CTA waits on counters that other CTAs advance: all must be resident
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return nt == 1 ? cudaLaunchKernelEx(&cfg, pass_kernel<1>, p) : cudaLaunchKernelEx(&cfg, pass_kernel<2>, p);
}

}  // namespace kvr
