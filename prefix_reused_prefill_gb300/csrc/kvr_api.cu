// C-ABI of libkvr: the slot table and the suffix-prefill driver.
//
// Host policy (goinfer, "Turn nine in under half a second", "How it works" and
// "Use it"): longest common prefix, the anti-theft rule, empty slot else LRU,
// truncation to the common length, reused-token count; --kv-sessions 0 turns
// reuse off; the memory check may grant fewer slots than requested.
// Device work is enqueued on the caller's stream; the library owns no device
// memory -- it carves the caller's arena and scratch buffers.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <string>
#include <tuple>
#include <vector>

#include <cudaTypedefs.h>

#include "kvr_internal.cuh"

using namespace kvr;

bool kvr::pdl_enabled() {
  static const bool on = [] {
    const char* v = getenv("KVR_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

namespace {

constexpr size_t kAlign = 256;
constexpr int kCounters = 16384;   // per-tile arrival counters of the fused GEMV epilogues
// then per (row tile, KV head) arrival counters of the split-KV attention's own merge
constexpr int kAttnCounters = 4096;
constexpr int kVerifyMaxRows = 64; // rows of one verify call
inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }

enum ProfClass { kProj = 0, kAttn = 1, kEpi = 2, kMatch = 3 };

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// int4 group-32 or K-quant: the 4-bit formats of the GEMV and the tcgen05 GEMM
bool packed4(const kvr_config& c) {
  return c.weight_format == KVR_WEIGHTS_INT4_G32 || c.weight_format == KVR_WEIGHTS_Q4K;
}
int weight_fmt(const kvr_config& c) { return c.weight_format == KVR_WEIGHTS_Q4K ? kFmtQ4K : kFmtInt4; }

bool valid_config(const kvr_config* c, std::string* why) {
  auto bad = [&](const char* m) { if (why) *why = m; return false; };
  if (!c) return bad("config is null");
  if (c->n_slots < 0 || c->n_slots > KVR_MAX_SLOTS) return bad("n_slots must be in [0, 16]");
  if (c->capacity <= 0 || c->capacity % kAttnKeys) return bad("capacity must be a positive multiple of 64");
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0)
    return bad("layer shape must be positive");
  if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c->n_q_heads % c->n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
  if (c->hidden % 8 || c->hidden > 8192) return bad("hidden must be a multiple of 8, at most 8192");
  if (!c->attn_only && (c->ffn <= 0 || c->ffn % 8)) return bad("ffn must be a positive multiple of 8");
  if (c->weight_format != KVR_WEIGHTS_BF16 && c->weight_format != KVR_WEIGHTS_INT4_G32 &&
      c->weight_format != KVR_WEIGHTS_Q4K)
    return bad("weight_format must be 0 (bf16), 1 (int4 g32) or 2 (q4k)");
  if (packed4(*c)) {
    if (c->hidden % kGemvKStep || (c->n_q_heads * c->head_dim) % kGemvKStep ||
        (!c->attn_only && c->ffn % kGemvKStep))
      return bad("int4 weights need every projection input width to be a multiple of 256");
  }
  if (c->max_rows <= 0) return bad("max_rows must be positive");
  if (c->max_rows > c->capacity) return bad("max_rows must not exceed capacity");
  if ((long long)c->max_rows * c->n_q_heads / c->n_kv_heads > (1 << 20)) return bad("max_rows too large");
  if (c->vocab < 0 || c->vocab > KVR_MAX_VOCAB) return bad("vocab must be in [0, 262144]");
  return true;
}

size_t slot_kv_bytes(const kvr_config* c) {
  return (size_t)c->n_layers * 2 * c->n_kv_heads * (size_t)c->capacity * c->head_dim * 2;
}

int qkv_cols(const kvr_config* c) { return (c->n_q_heads + 2 * c->n_kv_heads) * c->head_dim; }
int max_ldo(const kvr_config* c) {
  int v = std::max(qkv_cols(c), c->hidden);
  if (!c->attn_only) v = std::max(v, 2 * c->ffn);
  return v;
}

int attn_row_warps(int R) { return R <= 16 ? 1 : (R <= 32 ? 2 : 4); }

// Key splits of the split-KV kernel: about `target` CTAs, each with at least
// two 64-key blocks per consumer warp row, or one block per key-parallel warp
// (one row tile: four warps take alternate blocks, one CTA per SM).
int attn_nsplit(int Hkv, int R, int kend_max, int target) {
  const int rw = attn_row_warps(R);
  const int rt = (R + 16 * rw - 1) / (16 * rw);
  const int nb = (kend_max + kAttnKeys - 1) / kAttnKeys;
  int ns = (target + Hkv * rt - 1) / (Hkv * rt);
  ns = std::min(ns, std::max(1, rw == 1 ? nb / attn_key_warps(rw) : nb / 2));
  return std::max(1, std::min(ns, kMaxSplits));
}

struct ScratchLayout {
  size_t status, counters, prompt, slot_len, match_out, rope, h, a, q, o, z, part, opart, ml, best, next;
  size_t pass_layers, pass_done, pass_ss, pass_diag, total;
  size_t part_floats, opart_floats, ml_count;
};

ScratchLayout scratch_layout(const kvr_config* c) {
  ScratchLayout L{};
  const int S = std::max(c->n_slots, 1);
  const size_t M = c->max_rows, H = c->hidden, QD = (size_t)c->n_q_heads * c->head_dim;
  const size_t F = c->attn_only ? 0 : c->ffn;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + std::max<size_t>(bytes, 1)); return at; };
  L.status = take(64);
  L.counters = take((kCounters + kAttnCounters) * 4);
  L.prompt = take((size_t)c->capacity * 4);
  L.slot_len = take(KVR_MAX_SLOTS * 4);
  L.match_out = take((size_t)(S + 1) * S * 4);
  L.rope = take(M * (c->head_dim / 2) * 8);
  L.h = take(M * H * 4);
  L.a = take(M * H * 2);
  L.q = take(M * QD * 2);
  L.o = take(M * QD * 2);
  L.z = take(M * F * 2);
  // GEMV: [ksplit][tiles][32][128] tile-major partials (tiles round each segment up)
  L.part_floats = (size_t)kMaxKSplit * kGemvMaxCols * (max_ldo(c) + 3 * kGemvRows);
  if (packed4(*c))
    L.part_floats = std::max(L.part_floats, (size_t)kGemmMaxSplit * kGemmMaxTok *
                                                std::max(qkv_cols(c), c->hidden));
  // the output head's GEMV: up to three contributions per 128-row tile
  const size_t head_tiles = ((size_t)c->vocab + kGemvRows - 1) / kGemvRows;
  if (packed4(*c))
    L.part_floats = std::max(L.part_floats, head_tiles * 3 * kGemvMaxCols * kGemvRows);
  L.part = take(L.part_floats * 4);
  size_t worst = 0;
  const int G = c->n_q_heads / c->n_kv_heads;
  for (int m = 1; m <= c->max_rows; ++m) {
    const int ns = attn_nsplit(c->n_kv_heads, G * m, c->capacity, kSplitTargetCtas);
    if (ns > 1) worst = std::max(worst, (size_t)ns * m);
  }
  L.opart_floats = worst * c->n_q_heads * c->head_dim;
  L.ml_count = worst * c->n_q_heads;
  L.opart = take(L.opart_floats * 4);
  L.ml = take(L.ml_count * 8);
  L.best = take((size_t)kVerifyMaxRows * head_tiles * 8);
  L.next = take((size_t)kVerifyMaxRows * 4);
  // the persistent small-m pass: per-layer weight descriptors, completion
  // counters, per-tile sums of squares of its rows
  L.pass_layers = take((size_t)c->n_layers * sizeof(PassLayer));
  L.pass_done = take(((size_t)c->n_layers * kPassPhases + 8) * 4);
  L.pass_ss = take((size_t)kPassRows * ((H + kGemvRows - 1) / kGemvRows) * 4);
  L.pass_diag = take((size_t)kPassMaxCtas * 2 * 4);
  L.total = off;
  return L;
}

struct WKey {
  const void* p;
  int N, K, box, inner;
  bool operator<(const WKey& o) const {
    return std::tie(p, N, K, box, inner) < std::tie(o.p, o.N, o.K, o.box, o.inner);
  }
};
struct WMap {
  CUtensorMap w, s;
};

struct SlotState {
  bool occupied = false;
  std::vector<int32_t> tokens;
  unsigned long long stamp = 0;
};

struct EventPair {
  int cls;
  cudaEvent_t a, b;
};

}  // namespace

struct kvr_ctx {
  kvr_config cfg{};
  int requested = 0, granted = 0;
  bool reuse = true;
  int n_sms = 148;
  int fault = 0;  // 1 alloc, 2 launch, 3 capacity
  uint8_t* arena = nullptr;
  size_t arena_bytes = 0;
  int32_t* tok_mirror = nullptr;
  uint8_t* scratch = nullptr;
  ScratchLayout sl{};
  // scratch views
  int* status = nullptr;
  int* counters = nullptr;
  int32_t* prompt = nullptr;
  int* slot_len = nullptr;
  int32_t* match_out = nullptr;
  float2* rope = nullptr;
  RopeFreq rope_fr;   // theta^(-2j/d) in double, from the configuration
  float* h = nullptr;
  __nv_bfloat16 *a = nullptr, *q = nullptr, *o = nullptr, *z = nullptr;
  // the call's projections run on the tcgen05 GEMM, whose operands are fp16:
  // a, o and z then hold their bf16-rounded values in fp16
  bool act16 = false;
  // the persistent small-m pass: device layer table (and the host copy last
  // uploaded, pinned), completion counters and this context's call count
  PassLayer* pass_layers = nullptr;
  PassLayer* pass_host = nullptr;
  bool pass_uploaded = false;
  int* pass_done = nullptr;
  float* pass_ss = nullptr;
  int* pass_diag = nullptr;   // [kPassMaxCtas][2] where the pass's waits gave up
  unsigned pass_epoch = 0;
  bool use_pass = false;    // KVR_PASS=1 routes small m through the persistent pass
  float* part = nullptr;
  float* opart = nullptr;
  float2* ml = nullptr;
  float2* best = nullptr;   // output head: per row and tile, the largest logit and its index
  int32_t* next = nullptr;  // output head: per row, the argmax
  // TMA descriptors
  CUtensorMap tm_kv{}, tm_vt{}, tm_q{};
  CUtensorMap tm_a[6]{}, tm_o[6]{}, tm_z[6]{};
  std::map<WKey, WMap> wmaps;
  // slot table
  SlotState slots[KVR_MAX_SLOTS];
  unsigned long long clock = 0;
  // the match lengths read back by kvr_slot_match, [(slots + 1) * slots]; pinned,
  // so the read-back is one DMA straight into it
  int32_t* host_match = nullptr;
  size_t host_match_n = 0;
  // profiling
  bool prof = false;
  float* trace = nullptr;   // [n_layers + 1][max_rows][hidden] float32, or null
  bool force_gemv = false;  // KVR_FORCE_GEMV=1: keep every m on the GEMV path
  bool force_gemm = false;  // KVR_FORCE_GEMM=1: every m on the tcgen05 GEMM (a GEMV-free process)
  bool attn_combine = false; // KVR_ATTN_COMBINE=1: small-m split-KV partials merged by the combine launch
  int attn_splits = 0;      // KVR_ATTN_SPLITS=n: fixed key-split count of the tcgen05 attention
  std::vector<EventPair> pending;
  std::vector<cudaEvent_t> free_events;
  float prof_ms[4] = {0, 0, 0, 0};
  int prof_launches[4] = {0, 0, 0, 0};
  std::string err;
};

namespace {

// m rows of a 4-bit stack take the GEMV (else the tcgen05 GEMM)
bool gemv_path(const kvr_ctx* c, int m) {
  return c->force_gemv || (m <= kGemvMaxCols && !c->force_gemm);
}

int fail(kvr_ctx* c, int code, const char* fmt, ...) {
  if (c) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    c->err = buf;
  }
  return code;
}

int cuda_fail(kvr_ctx* c, cudaError_t e, const char* what) {
  return fail(c, KVR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

cudaEvent_t get_event(kvr_ctx* c) {
  if (!c->free_events.empty()) {
    cudaEvent_t e = c->free_events.back();
    c->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Brackets one launch with an event pair when profiling is on.
struct Timed {
  kvr_ctx* c;
  int cls;
  cudaStream_t st;
  cudaEvent_t a = nullptr;
  Timed(kvr_ctx* c_, int cls_, cudaStream_t st_) : c(c_), cls(cls_), st(st_) {
    c->prof_launches[cls]++;
    if (c->prof) {
      a = get_event(c);
      cudaEventRecord(a, st);
    }
  }
  ~Timed() {
    if (c->prof && a) {
      cudaEvent_t b = get_event(c);
      cudaEventRecord(b, st);
      c->pending.push_back({cls, a, b});
    }
  }
};

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* ptr, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle sw) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t es[2] = {1, 1};
  CUresult r = g_encode(m, dt, 2, const_cast<void*>(ptr), dims, strides, box, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// boxes of 8/16/32 rows (GEMV passes) and 64/128/256 rows (GEMM passes)
bool act_maps(CUtensorMap out[6], const void* buf, int K, int rows) {
  const int box[6] = {8, 16, 32, 64, 128, 256};
  for (int i = 0; i < 6; ++i)
    if (!encode_2d(&out[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, buf, K, rows, (uint64_t)K * 2, 64,
                   box[i], CU_TENSOR_MAP_SWIZZLE_128B))
      return false;
  return true;
}

// int4 weight (and scale) tensor maps: box of `box` rows x `inner` bytes (128: 128-byte
// swizzle, GEMV; 64: 64-byte swizzle, tcgen05 GEMM), cached per matrix.
const WMap* weight_map(kvr_ctx* c, const void* w, const void* s, int N, int K, int box = kGemvRows,
                       int inner = 128) {
  WKey key{w, N, K, box, inner};
  auto it = c->wmaps.find(key);
  if (it != c->wmaps.end()) return &it->second;
  WMap m;
  if (!encode_2d(&m.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, w, K / 2, N, K / 2, inner, box,
                 inner == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
    return nullptr;
  if (!encode_2d(&m.s, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, s, K / 32, N, (uint64_t)K / 32 * 2, 8,
                 box, CU_TENSOR_MAP_SWIZZLE_NONE))
    return nullptr;
  if (c->wmaps.size() > 4096) c->wmaps.clear();
  return &(c->wmaps[key] = m);
}

// ---------------------------------------------------------------------------
// projections
// ---------------------------------------------------------------------------
struct Seg {
  const void* w;
  const void* s;
  int N;
};

enum class Act { A, O, Z };

// Large-m passes on the tcgen05 GEMM; swiglu = 1 fuses silu(gate)*up into its
// epilogue; exact = 1 carries each weight as two fp16 terms (the QKV projection:
// q and k feed the softmax, which can amplify a weight's fp16 rounding).
template <class Epi>
int project_gemm(kvr_ctx* c, cudaStream_t st, const Seg* segs, int nseg, const CUtensorMap* tmx,
                 int K, int m, bool swiglu, bool exact, Epi epi) {
  GemmParams p;
  memset(&p, 0, sizeof p);
  p.K = K;
  p.kchunks = K / 128;
  p.status = c->status;
  p.part = c->part;
  p.z = c->z;
  p.z16 = 1;   // z feeds the down projection, on this GEMM as well
  p.F = c->cfg.ffn;
  int col = 0, tiles = 0;
  if (swiglu) {
    const WMap* g = weight_map(c, segs[0].w, segs[0].s, segs[0].N, K, 64, 64);
    const WMap* u = weight_map(c, segs[1].w, segs[1].s, segs[1].N, K, 64, 64);
    if (!g || !u) return fail(c, KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
    p.nseg = 1;
    p.seg[0].tw = g->w; p.seg[0].scales = static_cast<const __half*>(segs[0].s);
    p.seg[1].tw = u->w; p.seg[1].scales = static_cast<const __half*>(segs[1].s);
    p.seg[1].N = segs[1].N;
    p.seg[0].N = segs[0].N;
    p.seg[0].tiles = (segs[0].N + 63) / 64;
    tiles = p.seg[0].tiles;
    col = 2 * segs[0].N;
  } else {
    p.nseg = nseg;
    for (int i = 0; i < nseg; ++i) {
      const WMap* wm = weight_map(c, segs[i].w, segs[i].s, segs[i].N, K, 128, 64);
      if (!wm) return fail(c, KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
      GemmSeg& g = p.seg[i];
      g.tw = wm->w; g.scales = static_cast<const __half*>(segs[i].s);
      g.N = segs[i].N; g.col0 = col; g.tile0 = tiles; g.tiles = (segs[i].N + 127) / 128;
      col += segs[i].N;
      tiles += g.tiles;
    }
  }
  p.ldo = col;
  p.plane = (long long)kGemmMaxTok * p.ldo;
  p.swiglu = swiglu ? 1 : 0;
  p.exact = exact ? 1 : 0;
  p.fmt = weight_fmt(c->cfg);
  int ks = 1;
  if (!swiglu) {
    ks = (c->n_sms + tiles / 2) / std::max(tiles, 1);
    ks = std::max(1, std::min(ks, std::min(p.kchunks, kGemmMaxSplit)));
  }
  p.ksplit = ks;
  for (int t0 = 0; t0 < m; t0 += kGemmMaxTok) {
    const int mp = std::min(kGemmMaxTok, m - t0);
    p.t0 = t0;
    p.m = mp;
    p.n_tok = (mp + 15) / 16 * 16;
    p.xrows = p.n_tok <= 64 ? 64 : (p.n_tok <= 128 ? 128 : 256);
    p.tx = tmx[p.xrows == 64 ? 3 : (p.xrows == 128 ? 4 : 5)];
    cudaError_t e;
    {
      Timed t(c, kProj, st);
      e = launch_gemm_int4_tc(p, tiles, st);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "gemm_int4_tc launch");
    if (!swiglu) {
      Timed t(c, kEpi, st);
      e = epi(p.part, p.plane, p.ksplit, p.ldo, t0, mp);
      if (e != cudaSuccess) return cuda_fail(c, e, "epilogue launch");
    }
  }
  return KVR_OK;
}

// element offset of (slot, layer, K or V^T, head 0) in the arena
long long kv_offset(const kvr_ctx* c, int slot, int layer, int kind) {
  const kvr_config& k = c->cfg;
  return ((((long long)slot * k.n_layers + layer) * 2 + kind) * k.n_kv_heads) * (long long)k.capacity *
         k.head_dim;
}

// The epilogue the small-m int4 GEMV applies itself (see GemvEpi).
struct Fused {
  int epi = kGemvEpiResid;
  const RowMap* rows = nullptr;           // QKV
  long long k_off = 0, v_off = 0;         // QKV
  __nv_bfloat16* out = nullptr;           // Resid (last layer) / Cast
  const __nv_bfloat16* norm_gain = nullptr;  // Resid: RMSNorm the new rows into c->a
  float2* best = nullptr;                 // Argmax
  int fmt = -1;                           // WeightFmt; -1: the layers' format
};

// Small-m int4 passes: the GEMV with its fused epilogue.  A residual
// projection with a norm gain is followed by the row-wise RMSNorm launch that
// forms the next projection's input a.
int project_gemv_int4(kvr_ctx* c, cudaStream_t st, const Seg* segs, int nseg, const CUtensorMap* tmx,
                      int K, int m, const Fused& fz) {
  const kvr_config& cfg = c->cfg;
  const bool pair = fz.epi == kGemvEpiSwiglu;
  GemvParams p;
  memset(&p, 0, sizeof p);
  p.K = K;
  p.ksteps = K / kGemvKStep;
  p.status = c->status;
  p.part = c->part;
  p.epi = fz.epi;
  p.fmt = fz.fmt >= 0 ? fz.fmt : weight_fmt(cfg);
  p.counters = c->counters;
  int tiles = 0;
  if (pair) {
    const WMap* g = weight_map(c, segs[0].w, segs[0].s, segs[0].N, K, 64);
    const WMap* u = weight_map(c, segs[1].w, segs[1].s, segs[1].N, K, 64);
    if (!g || !u) return fail(c, KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
    p.nseg = 1;
    p.seg[0].tw = g->w; p.seg[0].ts = g->s; p.seg[0].N = segs[0].N;
    p.seg[1].tw = u->w; p.seg[1].ts = u->s; p.seg[1].N = segs[1].N;
    tiles = (segs[0].N + 63) / 64;
    p.seg[0].tiles = tiles;
  } else {
    p.nseg = nseg;
    int col = 0;
    for (int i = 0; i < nseg; ++i) {
      GemvSeg& g = p.seg[i];
      const WMap* wm = weight_map(c, segs[i].w, segs[i].s, segs[i].N, K);
      if (!wm) return fail(c, KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
      g.tw = wm->w;
      g.ts = wm->s;
      g.N = segs[i].N;
      g.col0 = col;
      g.tile0 = tiles;
      g.tiles = (segs[i].N + kGemvRows - 1) / kGemvRows;
      col += segs[i].N;
      tiles += g.tiles;
    }
  }
  if (tiles > kCounters) return fail(c, KVR_ERR_UNSUPPORTED, "projection has %d tiles (max %d)", tiles, kCounters);
  p.tiles = tiles;
  if (fz.rows) p.rows = *fz.rows;
  p.rope = c->rope;
  p.q = c->q;
  p.arena = reinterpret_cast<__nv_bfloat16*>(c->arena);
  p.k_off = fz.k_off;
  p.v_off = fz.v_off;
  p.cap = cfg.capacity;
  p.Hq = cfg.n_q_heads;
  p.Hkv = cfg.n_kv_heads;
  p.d = cfg.head_dim;
  p.h = c->h;
  p.H = cfg.hidden;
  p.out = fz.out;
  p.ldout = cfg.hidden;
  p.z = c->z;
  p.F = cfg.ffn;
  p.slot_stride = kv_offset(c, 1, 0, 0);
  p.best = fz.best;
  for (int c0 = 0; c0 < m; c0 += kGemvMaxCols) {
    const int mb = std::min(kGemvMaxCols, m - c0);
    p.c0 = c0;
    p.mb = mb;
    const int nt = mb <= 8 ? 1 : (mb <= 16 ? 2 : 4);
    // CTAs resident per SM (shared memory, registers): 2 up to 16 tokens, 1
    // beyond, and 1 where a variant's shared memory leaves no room for a second
    const int per_sm = std::max(1, gemv_int4_per_sm(nt, p.epi, p.fmt));
    p.tx = tmx[nt == 1 ? 0 : (nt == 2 ? 1 : 2)];
    // one resident wave of CTAs, each an equal run of (tile, k-step) units
    const int units = tiles * p.ksteps;
    int ctas = std::min(units, c->n_sms * per_sm);
    int maxc = 0;
    for (int tries = 0;; ++tries) {
      if (tries == 64) return fail(c, KVR_ERR_UNSUPPORTED, "no GEMV decomposition fits the scratch buffer");
      const int upc = units / ctas;                       // fewest units of a CTA
      maxc = (p.ksteps + upc - 1) / upc + 1;              // most contributors of a tile
      const int most_tiles = ((units + ctas - 1) / ctas + p.ksteps - 1) / p.ksteps + 1;
      const bool fits = (size_t)tiles * maxc * kGemvMaxCols * kGemvRows <= c->sl.part_floats;
      if (fits && most_tiles <= 16) break;
      if (!fits && ctas > 1) ctas = std::max(1, ctas * 3 / 4);
      else if (most_tiles > 16 && ctas < units) ctas = std::min(units, ctas * 2);
      else return fail(c, KVR_ERR_UNSUPPORTED, "no GEMV decomposition fits the scratch buffer");
    }
    p.ctas = ctas;
    p.maxc = maxc;
    p.ksplit = 1;
    cudaError_t e;
    {
      Timed t(c, kProj, st);
      e = launch_gemv_int4(p, nt, st);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "gemv_int4 launch");
  }
  if (fz.epi == kGemvEpiResid && fz.norm_gain) {
    Timed t(c, kEpi, st);
    const cudaError_t e = launch_norm(c->h, m, cfg.hidden, fz.norm_gain, cfg.rms_eps, c->a, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "norm launch");
  }
  return KVR_OK;
}

template <class Epi>
int project(kvr_ctx* c, cudaStream_t st, const Seg* segs, int nseg, Act act, int K, int m, Epi epi,
            const Fused& fz, bool swiglu = false, bool exact = false) {
  const kvr_config& cfg = c->cfg;
  const CUtensorMap* tmx = act == Act::A ? c->tm_a : (act == Act::O ? c->tm_o : c->tm_z);
  if (packed4(cfg) && gemv_path(c, m)) return project_gemv_int4(c, st, segs, nseg, tmx, K, m, fz);
  if (packed4(cfg)) return project_gemm(c, st, segs, nseg, tmx, K, m, swiglu, exact, epi);
  // bf16 weights: plain GEMV into partials, then the row-wise epilogue kernel
  GemvParams p;
  memset(&p, 0, sizeof p);
  p.nseg = nseg;
  p.K = K;
  p.status = c->status;
  int col = 0;
  for (int i = 0; i < nseg; ++i) {
    GemvSeg& g = p.seg[i];
    g.N = segs[i].N;
    g.col0 = col;
    g.wbf = static_cast<const __nv_bfloat16*>(segs[i].w);
    col += segs[i].N;
  }
  p.ldo = col;
  p.part = c->part;
  p.x = act == Act::A ? c->a : (act == Act::O ? c->o : c->z);
  p.ksplit = 1;
  p.plane = (long long)kGemvMaxCols * p.ldo;
  for (int c0 = 0; c0 < m; c0 += kGemvMaxCols) {
    const int mb = std::min(kGemvMaxCols, m - c0);
    p.c0 = c0;
    p.mb = mb;
    cudaError_t e;
    {
      Timed t(c, kProj, st);
      e = launch_gemv_bf16(p, col, st);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "gemv_bf16 launch");
    {
      Timed t(c, kEpi, st);
      e = epi(p.part, p.plane, p.ksplit, p.ldo, c0, mb);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "epilogue launch");
  }
  return KVR_OK;
}


// row of (slot, layer, K, head 0, position 0) in the [rows][head_dim] view of the arena
int k_row(const kvr_ctx* c, int slot, int layer) {
  const kvr_config& k = c->cfg;
  return (int)((((long long)slot * k.n_layers + layer) * 2) * k.n_kv_heads * (long long)k.capacity);
}

// row of (slot, layer, V^T, head 0, element 0) in the [rows][capacity] view of the arena
int vt_row(const kvr_ctx* c, int slot, int layer) {
  const kvr_config& k = c->cfg;
  return (int)((((long long)slot * k.n_layers + layer) * 2 + 1) * k.n_kv_heads * (long long)k.head_dim);
}

// Attention of one slot's rows (tokens tok0 .. tok0 + rows.m of the call; a
// batch runs one of these per conversation).
// The split-KV kernel with one row tile per CTA (rw == 1: four key-parallel
// warps) merges its own splits when a row tile has at most one row per warp
// (R <= 4): the last split of each (row tile, KV head) does it, so no combine
// launch follows.  With more rows each warp would merge them one after the
// other, and the combine launch (a warp per row) is faster (measured at 12
// and 16 rows: 2.57 / 2.63 ms per verify call against 2.50).
bool own_merge(const kvr_ctx* c, int rw, int row_tiles, int rows_per_tile) {
  return rw == 1 && rows_per_tile <= attn_key_warps(1) && !c->attn_combine &&
         (long long)row_tiles * c->cfg.n_kv_heads <= kAttnCounters;
}

int attention(kvr_ctx* c, cudaStream_t st, int slot, int layer, const RowMap& rows, int tok0 = 0) {
  const kvr_config& k = c->cfg;
  AttnParams p;
  memset(&p, 0, sizeof p);
  p.tkv = c->tm_kv;
  p.tvt = c->tm_vt;
  p.tq = c->tm_q;
  const long long qd = (long long)tok0 * k.n_q_heads * k.head_dim;
  p.q = c->q + qd;
  p.qrow0 = tok0 * k.n_q_heads;
  p.o = c->o + qd;
  p.opart = c->opart;
  p.ml = c->ml;
  p.rows = rows;
  p.Hq = k.n_q_heads;
  p.Hkv = k.n_kv_heads;
  p.G = k.n_q_heads / k.n_kv_heads;
  p.kbase = k_row(c, slot, layer);
  p.vtbase = vt_row(c, slot, layer);
  p.cap = k.capacity;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)k.head_dim);
  p.status = c->status;
  p.o16 = c->act16 ? 1 : 0;
  const int R = p.G * rows.m;
  const int kend = rows.P + rows.m;
  const bool tc = R > kAttnTcMinRows && !c->force_gemv;
  int ns;
  if (tc) {
    // tcgen05 path: 128-row tiles (one CTA per SM); split the keys as far as
    // one wave allows -- a partial second wave costs as much as a full one
    p.row_tiles = (R + 127) / 128;
    const int nb = (kend + kAttnTcKeys - 1) / kAttnTcKeys;
    ns = std::max(1, c->n_sms / (p.row_tiles * k.n_kv_heads));
    ns = std::max(1, std::min(std::min(ns, std::max(1, nb / 4)), kMaxSplits));
    if (c->attn_splits > 0) ns = std::min(c->attn_splits, std::min(nb, kMaxSplits));
  } else {
    const int rw = attn_row_warps(R);
    p.row_tiles = (R + 16 * rw - 1) / (16 * rw);
    // key-parallel warps (one row tile) run one CTA per SM: one wave of them
    ns = attn_nsplit(k.n_kv_heads, R, kend, rw == 1 ? c->n_sms : kSplitTargetCtas);
  }
  while (ns > 1 && (size_t)ns * rows.m * k.n_q_heads * k.head_dim > c->sl.opart_floats) --ns;
  p.nsplit = ns;
  p.counters = own_merge(c, tc ? 0 : attn_row_warps(R), p.row_tiles, R) ? c->counters + kCounters : nullptr;
  cudaError_t e;
  {
    Timed t(c, kAttn, st);
    e = tc ? launch_attention_tc(p, k.head_dim, st)
           : launch_attention(p, k.head_dim, attn_row_warps(R), st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "attention launch");
  if (ns > 1 && !p.counters) {
    Timed t(c, kAttn, st);
    e = launch_attn_combine(p, k.head_dim, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "attention combine launch");
  }
  return KVR_OK;
}

// Split-KV attention of several small conversations of a batch in one launch
// (and one combine): each CTA serves a row tile of one conversation over its
// own slot.  Every conversation takes the same split count (one wave of CTAs
// over all their tiles), at most half its key blocks.
int attention_batch(kvr_ctx* c, cudaStream_t st, int layer, const RowMap& rows, const int* bs, int nbs) {
  const kvr_config& k = c->cfg;
  AttnParams p;
  memset(&p, 0, sizeof p);
  p.tkv = c->tm_kv;
  p.tvt = c->tm_vt;
  p.tq = c->tm_q;
  p.q = c->q;
  p.o = c->o;
  p.opart = c->opart;
  p.ml = c->ml;
  p.rows.m = rows.m;
  p.Hq = k.n_q_heads;
  p.Hkv = k.n_kv_heads;
  p.G = k.n_q_heads / k.n_kv_heads;
  p.cap = k.capacity;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)k.head_dim);
  p.status = c->status;
  p.o16 = c->act16 ? 1 : 0;
  int rmax = 0;
  for (int i = 0; i < nbs; ++i) rmax = std::max(rmax, p.G * (rows.off[bs[i] + 1] - rows.off[bs[i]]));
  const int rw = attn_row_warps(rmax);
  int tiles = 0;
  for (int i = 0; i < nbs; ++i) {
    const int b = bs[i];
    AttnConv& cv = p.conv[i];
    cv.kbase = k_row(c, rows.slot[b], layer);
    cv.vtbase = vt_row(c, rows.slot[b], layer);
    cv.P = rows.pre[b];
    cv.m = rows.off[b + 1] - rows.off[b];
    cv.tok0 = rows.off[b];
    cv.tile0 = tiles;
    tiles += (p.G * cv.m + 16 * rw - 1) / (16 * rw);
  }
  p.n_conv = nbs;
  p.row_tiles = tiles;
  const int target = rw == 1 ? c->n_sms : kSplitTargetCtas;
  const int ns = std::max(1, (target + k.n_kv_heads * tiles - 1) / (k.n_kv_heads * tiles));
  for (int i = 0; i < nbs; ++i) {
    const int nb = (p.conv[i].P + p.conv[i].m + kAttnKeys - 1) / kAttnKeys;
    const int cap = rw == 1 ? nb / attn_key_warps(rw) : nb / 2;
    p.conv[i].nsplit = std::max(1, std::min(std::min(ns, std::max(1, cap)), kMaxSplits));
  }
  // the partials of every split conversation must fit the scratch
  auto need = [&]() {
    size_t f = 0;
    for (int i = 0; i < nbs; ++i)
      if (p.conv[i].nsplit > 1) f += (size_t)p.conv[i].nsplit * p.conv[i].m * k.n_q_heads * k.head_dim;
    return f;
  };
  while (need() > c->sl.opart_floats) {   // need() > 0: some conversation still splits
    int big = -1;
    for (int i = 0; i < nbs; ++i)
      if (p.conv[i].nsplit > 1 &&
          (big < 0 || p.conv[i].nsplit * p.conv[i].m > p.conv[big].nsplit * p.conv[big].m))
        big = i;
    --p.conv[big].nsplit;
  }
  long long at = 0;
  bool combine = false;
  for (int i = 0; i < nbs; ++i) {
    p.conv[i].part0 = at;
    if (p.conv[i].nsplit > 1) {
      at += (long long)p.conv[i].nsplit * p.conv[i].m * k.n_q_heads * k.head_dim;
      combine = true;
    }
    p.nsplit = std::max(p.nsplit, p.conv[i].nsplit);
  }
  p.counters = own_merge(c, rw, tiles, rmax) ? c->counters + kCounters : nullptr;
  cudaError_t e;
  {
    Timed t(c, kAttn, st);
    e = launch_attention(p, k.head_dim, rw, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "attention launch");
  if (combine && !p.counters) {
    Timed t(c, kAttn, st);
    e = launch_attn_combine(p, k.head_dim, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "attention combine launch");
  }
  return KVR_OK;
}

// ---------------------------------------------------------------------------
// the persistent small-m pass
// ---------------------------------------------------------------------------
// It serves a call with int4 group-32 weights, whole decoder layers, one slot,
// up to kPassRows rows (and G * rows <= kPassMaxAttnRows) and head_dim 128.
bool pass_fits(const kvr_ctx* c, const RowMap& rows) {
  const kvr_config& k = c->cfg;
  return c->use_pass && !c->force_gemv && !c->force_gemm && pass_ctas() > 0 &&
         k.weight_format == KVR_WEIGHTS_INT4_G32 && !k.attn_only && !rows.batch && rows.m <= kPassRows &&
         (k.n_q_heads / k.n_kv_heads) * rows.m <= kPassMaxAttnRows && k.head_dim == 128 &&
         k.hidden % kGemvRows == 0 && k.n_kv_heads <= pass_ctas();
}

// contributors of the most shared tile, and whether every CTA touches at most
// 16 tiles, for `tiles` tiles of `ks` units over min(ctas, units) CTAs (the
// split of k_pass.cu)
bool pass_split(int tiles, int ks, int ctas, int* maxc) {
  const long long units = (long long)tiles * ks;
  ctas = (int)std::min<long long>(ctas, units);
  auto owner = [&](long long u) { return (int)(((u + 1) * ctas - 1) / units); };
  int mc = 1;
  for (int t = 0; t < tiles; ++t) mc = std::max(mc, owner((long long)t * ks + ks - 1) - owner((long long)t * ks) + 1);
  for (int b = 0; b < ctas; ++b) {
    const long long u0 = b * units / ctas, u1 = (b + 1) * units / ctas;
    if (u1 > u0 && (u1 - 1) / ks - u0 / ks + 1 > 16) return false;
  }
  *maxc = mc;
  return true;
}

int run_pass(kvr_ctx* c, const RowMap& rows, const void* hidden, const kvr_layer_weights* w, void* out,
             cudaStream_t st, const __nv_bfloat16* head_gain) {
  const kvr_config& k = c->cfg;
  const int L = k.n_layers, H = k.hidden, F = k.ffn, d = k.head_dim;
  const int Hq = k.n_q_heads, Hkv = k.n_kv_heads, m = rows.m;
  const int ctas = pass_ctas();
  // per-layer weight descriptors (the cached tensor maps), uploaded when they change
  std::vector<PassLayer> tab(L);
  for (int l = 0; l < L; ++l) {
    const kvr_layer_weights& W = w[l];
    const void* ws[7] = {W.wq, W.wk, W.wv, W.wo, W.wg, W.wu, W.wd};
    const void* ss[7] = {W.sq, W.sk, W.sv, W.so, W.sg, W.su, W.sd};
    const int N[7] = {Hq * d, Hkv * d, Hkv * d, H, F, F, H};
    const int K[7] = {H, H, H, Hq * d, H, H, F};
    PassLayer& T = tab[l];
    memset(&T, 0, sizeof T);
    for (int i = 0; i < 7; ++i) {
      const WMap* wm = weight_map(c, ws[i], ss[i], N[i], K[i], (i == 4 || i == 5) ? 64 : kGemvRows);
      if (!wm) return fail(c, KVR_ERR_CUDA, "cuTensorMapEncodeTiled failed for a weight matrix");
      T.tw[i] = wm->w;
      T.ts[i] = wm->s;
    }
    T.norm_attn = static_cast<const __nv_bfloat16*>(W.norm_attn);
    T.norm_ffn = static_cast<const __nv_bfloat16*>(W.norm_ffn);
  }
  const size_t tab_bytes = (size_t)L * sizeof(PassLayer);
  cudaError_t e = cudaSuccess;
  if (!c->pass_uploaded || memcmp(c->pass_host, tab.data(), tab_bytes) != 0) {
    // the pinned copy may still feed an earlier upload
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(c, e, "pass table upload");
    memcpy(c->pass_host, tab.data(), tab_bytes);
    e = cudaMemcpyAsync(c->pass_layers, c->pass_host, tab_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "pass table upload");
    c->pass_uploaded = true;
  }
  PassParams p;
  memset(&p, 0, sizeof p);
  p.layers = c->pass_layers;
  p.L = L; p.H = H; p.F = F; p.Hq = Hq; p.Hkv = Hkv; p.d = d; p.G = Hq / Hkv; p.cap = k.capacity;
  p.m = m;
  p.rows = rows;
  p.slot = rows.slot[0];
  p.tkv = c->tm_kv;
  p.tvt = c->tm_vt;
  p.arena = reinterpret_cast<__nv_bfloat16*>(c->arena);
  p.kv_slot = kv_offset(c, rows.slot[0], 0, 0);
  p.kbase0 = k_row(c, rows.slot[0], 0);
  p.vtbase0 = vt_row(c, rows.slot[0], 0);
  p.ctas = ctas;
  const int ksH = H / kGemvKStep, ksQ = Hq * d / kGemvKStep, ksF = F / kGemvKStep;
  const int tq = (Hq * d + kGemvRows - 1) / kGemvRows + 2 * ((Hkv * d + kGemvRows - 1) / kGemvRows);
  const int th = (H + kGemvRows - 1) / kGemvRows, tgu = (F + 63) / 64;
  const int tiles[kPassPhases] = {tq, 0, th, tgu, th};
  const int ks[kPassPhases] = {ksH, 0, ksQ, ksH, ksF};
  for (int ph = 0; ph < kPassPhases; ++ph) {
    if (ph == 1) continue;
    if (tiles[ph] > kCounters || !pass_split(tiles[ph], ks[ph], ctas, &p.maxc[ph]) ||
        (size_t)tiles[ph] * p.maxc[ph] * kGemvMaxCols * kGemvRows > c->sl.part_floats)
      return fail(c, KVR_ERR_UNSUPPORTED, "no split of the small-m pass fits its buffers");
  }
  p.nb = (rows.P + m + kAttnKeys - 1) / kAttnKeys;
  p.nsplit = std::max(1, std::min(std::min(ctas / Hkv, p.nb), kMaxSplits));   // the merge holds 64
  if (c->attn_splits > 0) p.nsplit = std::max(1, std::min(c->attn_splits, p.nsplit));
  while (p.nsplit > 1 && ((size_t)Hkv * p.nsplit * kPassMaxAttnRows * d > c->sl.opart_floats ||
                          (size_t)Hkv * p.nsplit * kPassMaxAttnRows > c->sl.ml_count))
    --p.nsplit;
  if ((size_t)Hkv * p.nsplit * kPassMaxAttnRows * d > c->sl.opart_floats)
    return fail(c, KVR_ERR_UNSUPPORTED, "attention partials of the small-m pass do not fit");
  p.hidden = static_cast<const __nv_bfloat16*>(hidden);
  p.h = c->h;
  p.ss = c->pass_ss;
  p.nss = H / kGemvRows;
  p.rope = c->rope;
  p.q = c->q;
  p.o = c->o;
  p.z = c->z;
  p.part = c->part;
  p.opart = c->opart;
  p.ml = c->ml;
  p.tile_cnt = c->counters;
  p.head_cnt = c->counters + kCounters;
  p.done = c->pass_done;
  // completion counters grow by one call's count per call; restart them
  // before the products could overflow
  if (c->pass_epoch >= (1u << 20)) {
    e = cudaMemsetAsync(c->pass_done, 0, ((size_t)L * kPassPhases + 8) * 4, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "pass counter reset");
    c->pass_epoch = 0;
  }
  p.epoch = ++c->pass_epoch;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.head_gain = head_gain;
  p.a_head = c->a;
  p.trace = c->trace;
  p.trace_rows = k.max_rows;
  p.diag = c->pass_diag;
  p.eps = k.rms_eps;
  p.scale_log2 = 1.4426950408889634f / sqrtf((float)d);
  p.status = c->status;
  c->act16 = false;
  {
    Timed t(c, kEpi, st);
    e = launch_rope_table(rows, d, c->rope_fr, c->rope, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "rope table launch");
  {
    Timed t(c, kProj, st);
    e = launch_pass(p, m <= 8 ? 1 : 2, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "small-m pass launch");
  return KVR_OK;
}

// The layer stack for the rows of one call.
// out (bf16 [m][hidden]) may be null; head_gain: RMSNorm the last layer's rows
// with it into c->a (the output head's input)
int run_stack(kvr_ctx* c, const RowMap& rows, const void* hidden,
              const kvr_layer_weights* w, void* out, cudaStream_t st,
              const __nv_bfloat16* head_gain = nullptr) {
  if (pass_fits(c, rows)) return run_pass(c, rows, hidden, w, out, st, head_gain);
  const kvr_config& k = c->cfg;
  const int m = rows.m, H = k.hidden, d = k.head_dim;
  const int Hq = k.n_q_heads, Hkv = k.n_kv_heads, F = k.ffn;
  cudaError_t e;
  c->act16 = packed4(k) && !gemv_path(c, m);
  {
    // the rows' RoPE table and the first RMSNorm in one launch; attention-only
    // layers take the input rows as they are (no norm)
    Timed t(c, kEpi, st);
    e = launch_embed(static_cast<const __nv_bfloat16*>(hidden), m, H,
                     k.attn_only ? nullptr : static_cast<const __nv_bfloat16*>(w[0].norm_attn), k.rms_eps,
                     c->h, c->a, c->act16, rows, d, c->rope_fr, c->rope, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "embed launch");
  }
  auto trace = [&](int entry) -> cudaError_t {
    if (!c->trace || k.attn_only) return cudaSuccess;
    return cudaMemcpyAsync(c->trace + (size_t)entry * k.max_rows * H, c->h, (size_t)m * H * 4,
                           cudaMemcpyDeviceToDevice, st);
  };
  e = trace(0);
  if (e != cudaSuccess) return cuda_fail(c, e, "trace copy");
  __nv_bfloat16* arena = reinterpret_cast<__nv_bfloat16*>(c->arena);
  for (int l = 0; l < k.n_layers; ++l) {
    const kvr_layer_weights& W = w[l];
    const bool last = l == k.n_layers - 1;
    // Q, K, V (+ RoPE, append)
    {
      Seg segs[3] = {{W.wq, W.sq, Hq * d}, {W.wk, W.sk, Hkv * d}, {W.wv, W.sv, Hkv * d}};
      // K/V of slot 0 of this layer; each row adds its slot's stride
      const long long koff = kv_offset(c, 0, l, 0), voff = kv_offset(c, 0, l, 1);
      const long long sstride = kv_offset(c, 1, 0, 0);
      Fused fz;
      fz.epi = kGemvEpiQKV;
      fz.rows = &rows;
      fz.k_off = koff;
      fz.v_off = voff;
      int rc = project(c, st, segs, 3, Act::A, H, m, [&](const float* part, long long plane, int ks,
                                                          int ldo, int c0, int mb) {
        return launch_epi_qkv(part, plane, ks, ldo, c0, mb, rows, Hq, Hkv, d, c->rope, c->q, arena,
                              koff, voff, sstride, k.capacity, st);
      }, fz, /*swiglu=*/false, /*exact=*/true);
      if (rc) return rc;
    }
    int rc = KVR_OK;
    if (!rows.batch) {
      rc = attention(c, st, rows.slot[0], l, rows);
    } else {
      // conversations with many rows take the tcgen05 kernel one by one; the
      // rest share one split-KV launch
      int small[KVR_MAX_BRANCHES], n_small = 0;
      for (int b = 0; b < rows.n_branch && !rc; ++b) {
        RowMap one;
        memset(&one, 0, sizeof one);
        one.P = rows.pre[b];
        one.m = rows.off[b + 1] - rows.off[b];
        one.n_branch = 1;
        one.off[1] = one.m;
        one.slot[0] = rows.slot[b];
        if ((k.n_q_heads / k.n_kv_heads) * one.m > kAttnTcMinRows && !c->force_gemv)
          rc = attention(c, st, rows.slot[b], l, one, rows.off[b]);
        else
          small[n_small++] = b;
      }
      if (!rc && n_small) rc = attention_batch(c, st, l, rows, small, n_small);
    }
    if (rc) return rc;
    // O projection
    {
      Seg so = {W.wo, W.so, H};
      if (k.attn_only) {
        __nv_bfloat16* dst = last ? static_cast<__nv_bfloat16*>(out) : c->a;
        Fused fz;
        fz.epi = kGemvEpiCast;
        fz.out = dst;
        rc = project(c, st, &so, 1, Act::O, Hq * d, m,
                     [&](const float* part, long long plane, int ks, int ldo, int c0, int mb) {
                       return launch_epi_cast(part, plane, ks, ldo, c0, mb, H, dst, c->act16 && !last, st);
                     }, fz);
        if (rc) return rc;
        continue;
      }
      Fused fz;
      fz.epi = kGemvEpiResid;
      fz.norm_gain = static_cast<const __nv_bfloat16*>(W.norm_ffn);
      rc = project(c, st, &so, 1, Act::O, Hq * d, m,
                   [&](const float* part, long long plane, int ks, int ldo, int c0, int mb) {
                     return launch_epi_resid(part, plane, ks, ldo, c0, mb, H, c->h,
                                             static_cast<const __nv_bfloat16*>(W.norm_ffn),
                                             k.rms_eps, c->a, c->act16, nullptr, st);
                   }, fz);
      if (rc) return rc;
    }
    // gate | up -> SwiGLU
    {
      Seg gu[2] = {{W.wg, W.sg, F}, {W.wu, W.su, F}};
      Fused fz;
      fz.epi = kGemvEpiSwiglu;
      rc = project(c, st, gu, 2, Act::A, H, m,
                   [&](const float* part, long long plane, int ks, int ldo, int c0, int mb) {
                     return launch_epi_swiglu(part, plane, ks, ldo, c0, mb, F, c->z, st);
                   },
                   fz, /*swiglu=*/true);
      if (rc) return rc;
    }
    // down + residual, then the next layer's attention norm (the output head's
    // norm after the last layer), and the output
    {
      Seg sd = {W.wd, W.sd, H};
      const __nv_bfloat16* gain = last ? head_gain : static_cast<const __nv_bfloat16*>(w[l + 1].norm_attn);
      Fused fz;
      fz.epi = kGemvEpiResid;
      fz.norm_gain = gain;
      fz.out = last ? static_cast<__nv_bfloat16*>(out) : nullptr;
      rc = project(c, st, &sd, 1, Act::Z, F, m,
                   [&](const float* part, long long plane, int ks, int ldo, int c0, int mb) {
                     // the output head's input stays bf16 (the head runs on the GEMV)
                     return launch_epi_resid(part, plane, ks, ldo, c0, mb, H, c->h, gain, k.rms_eps,
                                             gain ? c->a : nullptr, c->act16 && !last,
                                             last ? static_cast<__nv_bfloat16*>(out) : nullptr, st);
                   }, fz);
      if (rc) return rc;
      e = trace(l + 1);
      if (e != cudaSuccess) return cuda_fail(c, e, "trace copy");
    }
  }
  return KVR_OK;
}

bool weights_ok(const kvr_ctx* c, const kvr_layer_weights* w) {
  if (!w) return false;
  const bool i4 = packed4(c->cfg);
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    const kvr_layer_weights& W = w[l];
    const void* need[] = {W.wq, W.wk, W.wv, W.wo};
    for (const void* p : need)
      if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return false;
    if (i4) {
      const void* sc[] = {W.sq, W.sk, W.sv, W.so};
      for (const void* p : sc)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return false;
    }
    if (!c->cfg.attn_only) {
      const void* ff[] = {W.wg, W.wu, W.wd, W.norm_attn, W.norm_ffn};
      for (const void* p : ff)
        if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return false;
      if (i4) {
        const void* sf[] = {W.sg, W.su, W.sd};
        for (const void* p : sf)
          if (!p || (reinterpret_cast<uintptr_t>(p) & 15)) return false;
      }
    }
  }
  return true;
}

void touch(kvr_ctx* c, int s) { c->slots[s].stamp = ++c->clock; }

int upload_tokens(kvr_ctx* c, int slot, int at, const int32_t* toks, int n, cudaStream_t st) {
  if (n <= 0) return KVR_OK;
  cudaError_t e = cudaMemcpyAsync(c->tok_mirror + (size_t)slot * c->cfg.capacity + at, toks,
                                  (size_t)n * 4, cudaMemcpyHostToDevice, st);
  return e == cudaSuccess ? KVR_OK : cuda_fail(c, e, "token mirror upload");
}

int prefill_common(kvr_ctx* c, int slot, const int32_t* tokens, int m, const void* hidden,
                   const kvr_layer_weights* w, void* out, void* stream, int max_m,
                   const __nv_bfloat16* head_gain = nullptr) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slot);
  if (!tokens || !hidden || (!out && !head_gain) || m <= 0)
    return fail(c, KVR_ERR_ARG, "null pointer or m <= 0");
  if (m > max_m) return fail(c, KVR_ERR_ARG, "m = %d exceeds %d for this call", m, max_m);
  if (((uintptr_t)hidden & 15) || ((uintptr_t)out & 15)) return fail(c, KVR_ERR_ARG, "hidden/out must be 16-byte aligned");
  if (!weights_ok(c, w)) return fail(c, KVR_ERR_ARG, "missing or misaligned weight pointer");
  const int p0 = (int)c->slots[slot].tokens.size();
  if (m > c->cfg.max_rows || p0 + m > c->cfg.capacity || c->fault == 3)
    return fail(c, KVR_ERR_CAPACITY, "slot %d: %d + %d rows exceed capacity %d (max_rows %d)", slot,
                p0, m, c->cfg.capacity, c->cfg.max_rows);
  if (c->fault == 2) return fail(c, KVR_ERR_FAULT, "injected launch fault");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  RowMap rows;
  memset(&rows, 0, sizeof rows);
  rows.P = p0;
  rows.m = m;
  rows.n_branch = 1;
  rows.off[0] = 0;
  rows.off[1] = m;
  rows.slot[0] = slot;
  int rc = run_stack(c, rows, hidden, w, out, st, head_gain);
  if (rc) return rc;
  rc = upload_tokens(c, slot, p0, tokens, m, st);
  if (rc) return rc;
  SlotState& S = c->slots[slot];
  S.occupied = true;
  S.tokens.insert(S.tokens.end(), tokens, tokens + m);
  touch(c, slot);
  return KVR_OK;
}

// ---------------------------------------------------------------- output head
int head_check(kvr_ctx* c, const kvr_head_weights* head, const void* next_tokens, const void* accepted) {
  const kvr_config& k = c->cfg;
  if (!head || !next_tokens || !accepted) return fail(c, KVR_ERR_ARG, "null head or result pointer");
  if (!packed4(k) || k.attn_only)
    return fail(c, KVR_ERR_UNSUPPORTED, "the output head needs int4 weights and the full decoder layer");
  if (head->vocab <= 0 || head->vocab > k.vocab)
    return fail(c, KVR_ERR_ARG, "head vocab %d outside [1, %d] (the configured vocab)", head->vocab, k.vocab);
  for (const void* q : {head->norm, head->w, head->s})
    if (!q || (reinterpret_cast<uintptr_t>(q) & 15)) return fail(c, KVR_ERR_ARG, "missing or misaligned head pointer");
  return KVR_OK;
}

// logits = a * lm^T over the m normed rows in c->a, each tile's best, each
// row's argmax, read back to next_tokens; synchronises the stream
int head_decide(kvr_ctx* c, cudaStream_t st, int m, const kvr_head_weights* head, int32_t* next_tokens) {
  Seg seg = {head->w, head->s, head->vocab};
  Fused fz;
  fz.epi = kGemvEpiArgmax;
  fz.fmt = kFmtInt4;   // the head is int4 group-32 in every configuration
  fz.best = c->best;
  int rc = project_gemv_int4(c, st, &seg, 1, c->tm_a, c->cfg.hidden, m, fz);
  if (rc) return rc;
  cudaError_t e;
  {
    Timed t(c, kEpi, st);
    e = launch_head_argmax(c->best, (head->vocab + kGemvRows - 1) / kGemvRows, m, c->next, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "head argmax launch");
  e = cudaMemcpyAsync(next_tokens, c->next, (size_t)m * 4, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(c, e, "next-token readback");
  return kvr_sync_status(c, st);
}

// greedy acceptance of one conversation's rows [t0, d1 .. dk]
int greedy_accept(const int32_t* tokens, const int32_t* next, int m) {
  int a = 0;
  while (a + 1 < m && tokens[a + 1] == next[a]) ++a;
  return a;
}

// ---------------------------------------------------------------- slot policy
// The slot choice of goinfer "How it works" applied to the match kernel's
// result res ([S][S+1]: res[s][S] = LCP of slot s with the prompt, res[a][b]
// for a < b = LCP of slots a and b): the longest match wins if it is longer
// than what that slot shares with any other occupied slot (and, with an empty
// slot free, if it would not cut its conversation back); otherwise the lowest
// empty slot, else the least recently used one, starts from zero.  The chosen
// slot keeps min(match, n - 1) tokens and is touched.
void apply_slot_policy(kvr_ctx* c, const int32_t* res, int n, int* slot, int* reused) {
  const int S = c->granted;
  const int W = S + 1;
  auto pair = [&](int a, int b) { return a < b ? res[a * W + b] : res[b * W + a]; };
  int l[KVR_MAX_SLOTS];
  int best = -1;
  bool any_empty = false;
  for (int s = 0; s < S; ++s) {
    l[s] = c->slots[s].occupied ? res[s * W + S] : 0;
    if (!c->slots[s].occupied) any_empty = true;
    if (c->slots[s].occupied && (best < 0 || l[s] > l[best])) best = s;
  }
  bool accept = best >= 0 && l[best] > 0;
  if (accept && c->cfg.match_threshold) {
    int o = 0;
    for (int t = 0; t < S; ++t)
      if (t != best && c->slots[t].occupied) o = std::max(o, pair(best, t));
    accept = l[best] > o;
    if (accept && any_empty && l[best] < (int)c->slots[best].tokens.size()) accept = false;
  }
  if (accept) {
    const int r = std::min(l[best], n - 1);
    c->slots[best].tokens.resize(r);
    touch(c, best);
    *slot = best;
    *reused = r;
    return;
  }
  int pick = -1;
  for (int s = 0; s < S && pick < 0; ++s)
    if (!c->slots[s].occupied) pick = s;
  if (pick < 0) {
    pick = 0;
    for (int s = 1; s < S; ++s)
      if (c->slots[s].stamp < c->slots[pick].stamp) pick = s;
  }
  c->slots[pick].occupied = true;
  c->slots[pick].tokens.clear();
  touch(c, pick);
  *slot = pick;
  *reused = 0;
}

// n_slots = 0 ("0 turns reuse off"): one working slot, cleared by every match
void match_without_reuse(kvr_ctx* c, int* slot, int* reused) {
  c->slots[0].occupied = true;
  c->slots[0].tokens.clear();
  touch(c, 0);
  *slot = 0;
  *reused = 0;
}

// ---------------------------------------------------------------- spill/restore
struct SpillHeader {
  char magic[8];      // "KVRSLOT1"
  uint64_t hash;      // kvr_config_hash of the writer
  uint64_t bytes;     // size of the whole record
  int32_t len, n_layers, n_kv_heads, head_dim;
  uint8_t reserved[24];
};
static_assert(sizeof(SpillHeader) == 64, "spill header is 64 bytes");
constexpr char kSpillMagic[8] = {'K', 'V', 'R', 'S', 'L', 'O', 'T', '1'};

struct SpillLayout {
  size_t tokens, kv, layer_bytes, half_bytes, total;
};

SpillLayout spill_layout(int len, int n_layers, int hkv, int d) {
  SpillLayout L;
  L.tokens = sizeof(SpillHeader);
  L.kv = L.tokens + align_up((size_t)len * 4, 16);
  L.half_bytes = (size_t)hkv * len * d * 2;   // K or V^T of one layer
  L.layer_bytes = 2 * L.half_bytes;
  L.total = L.kv + (size_t)n_layers * L.layer_bytes;
  return L;
}

uint64_t fnv1a_words(const uint32_t* w, int n, uint64_t tag) {
  uint64_t h = 0xcbf29ce484222325ull;
  auto eat = [&](uint8_t b) { h = (h ^ b) * 0x100000001b3ull; };
  for (int i = 0; i < n; ++i)
    for (int k = 0; k < 4; ++k) eat((uint8_t)(w[i] >> (8 * k)));
  for (int k = 0; k < 8; ++k) eat((uint8_t)(tag >> (8 * k)));
  return h;
}

uint32_t float_word(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

// one 2-D copy per layer for K ([Hkv] blocks of len*d) and one for V^T
// ([Hkv*d] rows of len); to_host picks the direction
cudaError_t copy_slot_kv(kvr_ctx* c, int slot, int len, uint8_t* host, bool to_host, cudaStream_t st) {
  const kvr_config& k = c->cfg;
  const size_t cap = k.capacity, d = k.head_dim, hkv = k.n_kv_heads;
  const SpillLayout L = spill_layout(len, k.n_layers, k.n_kv_heads, k.head_dim);
  if (len == 0) return cudaSuccess;
  uint8_t* arena = c->arena;
  for (int l = 0; l < k.n_layers; ++l) {
    uint8_t* kd = arena + kv_offset(c, slot, l, 0) * 2;
    uint8_t* vd = arena + kv_offset(c, slot, l, 1) * 2;
    uint8_t* kh = host + L.kv + l * L.layer_bytes;
    uint8_t* vh = kh + L.half_bytes;
    const size_t kw = (size_t)len * d * 2, vw = (size_t)len * 2;
    cudaError_t e;
    if (to_host) {
      e = cudaMemcpy2DAsync(kh, kw, kd, cap * d * 2, kw, hkv, cudaMemcpyDeviceToHost, st);
      if (e == cudaSuccess) e = cudaMemcpy2DAsync(vh, vw, vd, cap * 2, vw, hkv * d, cudaMemcpyDeviceToHost, st);
    } else {
      e = cudaMemcpy2DAsync(kd, cap * d * 2, kh, kw, kw, hkv, cudaMemcpyHostToDevice, st);
      if (e == cudaSuccess) e = cudaMemcpy2DAsync(vd, cap * 2, vh, vw, vw, hkv * d, cudaMemcpyHostToDevice, st);
    }
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

int batch_common(kvr_ctx* c, int n_seq, const int* slots, const int* lens, const int32_t* tokens,
                 const void* hidden, const kvr_layer_weights* w, void* out, void* stream, int max_m,
                 const __nv_bfloat16* head_gain) {
  if (!c) return KVR_ERR_ARG;
  if (n_seq < 1 || n_seq > KVR_MAX_BRANCHES || !slots || !lens || !tokens || !hidden || (!out && !head_gain))
    return fail(c, KVR_ERR_ARG, "bad batch arguments");
  if (((uintptr_t)hidden & 15) || ((uintptr_t)out & 15)) return fail(c, KVR_ERR_ARG, "hidden/out must be 16-byte aligned");
  if (!weights_ok(c, w)) return fail(c, KVR_ERR_ARG, "missing or misaligned weight pointer");
  RowMap rows;
  memset(&rows, 0, sizeof rows);
  rows.batch = 1;
  rows.n_branch = n_seq;
  int total = 0;
  for (int j = 0; j < n_seq; ++j) {
    const int s = slots[j];
    if (s < 0 || s >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", s);
    for (int i = 0; i < j; ++i)
      if (slots[i] == s) return fail(c, KVR_ERR_ARG, "slot %d appears twice in the batch", s);
    if (lens[j] <= 0) return fail(c, KVR_ERR_ARG, "conversation %d has %d rows", j, lens[j]);
    rows.slot[j] = s;
    rows.pre[j] = (int)c->slots[s].tokens.size();
    rows.off[j] = total;
    total += lens[j];
    if (rows.pre[j] + lens[j] > c->cfg.capacity || c->fault == 3)
      return fail(c, KVR_ERR_CAPACITY, "slot %d: %d + %d rows exceed capacity %d", s, rows.pre[j], lens[j],
                  c->cfg.capacity);
  }
  rows.off[n_seq] = total;
  rows.m = total;
  if (total > c->cfg.max_rows) return fail(c, KVR_ERR_CAPACITY, "%d rows exceed max_rows %d", total, c->cfg.max_rows);
  if (total > max_m) return fail(c, KVR_ERR_ARG, "%d rows exceed %d for this call", total, max_m);
  if (c->fault == 2) return fail(c, KVR_ERR_FAULT, "injected launch fault");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int rc = run_stack(c, rows, hidden, w, out, st, head_gain);
  if (rc) return rc;
  for (int j = 0; j < n_seq; ++j) {
    rc = upload_tokens(c, slots[j], rows.pre[j], tokens + rows.off[j], lens[j], st);
    if (rc) return rc;
  }
  for (int j = 0; j < n_seq; ++j) {
    SlotState& S = c->slots[slots[j]];
    S.occupied = true;
    S.tokens.insert(S.tokens.end(), tokens + rows.off[j], tokens + rows.off[j + 1]);
    touch(c, slots[j]);
  }
  return KVR_OK;
}

}  // namespace

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

size_t kvr_arena_bytes(const kvr_config* cfg, int n_slots) {
  if (!valid_config(cfg, nullptr) || n_slots <= 0) return 0;
  return (size_t)n_slots * (slot_kv_bytes(cfg) + (size_t)cfg->capacity * 4);
}

size_t kvr_scratch_bytes(const kvr_config* cfg) {
  if (!valid_config(cfg, nullptr)) return 0;
  return scratch_layout(cfg).total;
}

int kvr_ctx_create(const kvr_config* cfg, void* kv_arena, size_t arena_bytes, void* scratch,
                   size_t scratch_bytes, kvr_ctx** out) {
  if (!out) return KVR_ERR_ARG;
  *out = nullptr;
  std::string why;
  if (!valid_config(cfg, &why)) return KVR_ERR_ARG;
  if (!kv_arena || !scratch || ((uintptr_t)kv_arena & 255) || ((uintptr_t)scratch & 255))
    return KVR_ERR_ARG;
  kvr_ctx* c = new kvr_ctx();
  c->cfg = *cfg;
  const char* f = getenv("KVR_FAULT");
  if (f) {
    if (!strcmp(f, "alloc")) c->fault = 1;
    else if (!strcmp(f, "launch")) c->fault = 2;
    else if (!strcmp(f, "capacity")) c->fault = 3;
  }
  if (c->fault == 1) {
    delete c;
    return KVR_ERR_FAULT;
  }
  const char* fg = getenv("KVR_FORCE_GEMV");
  c->force_gemv = fg && fg[0] == '1';
  const char* fm = getenv("KVR_FORCE_GEMM");
  c->force_gemm = fm && fm[0] == '1';
  const char* ac = getenv("KVR_ATTN_COMBINE");
  c->attn_combine = ac && ac[0] == '1';
  const char* as = getenv("KVR_ATTN_SPLITS");
  c->attn_splits = as ? atoi(as) : 0;
  // the persistent pass is opt-in: measured on the 36-layer 4096-wide stack it
  // ties the per-step launches at one row and trails them from two rows on
  const char* ps = getenv("KVR_PASS");
  c->use_pass = ps && ps[0] == '1';
  c->requested = cfg->n_slots;
  c->reuse = cfg->n_slots > 0;
  const int want = std::max(cfg->n_slots, 1);
  const size_t per = slot_kv_bytes(cfg) + (size_t)cfg->capacity * 4;
  c->granted = (int)std::min<size_t>(want, arena_bytes / per);
  c->sl = scratch_layout(cfg);
  if (c->granted < 1 || scratch_bytes < c->sl.total) {
    delete c;
    return KVR_ERR_CAPACITY;
  }
  c->arena = static_cast<uint8_t*>(kv_arena);
  c->arena_bytes = arena_bytes;
  c->tok_mirror = reinterpret_cast<int32_t*>(c->arena + (size_t)c->granted * slot_kv_bytes(cfg));
  c->scratch = static_cast<uint8_t*>(scratch);
  uint8_t* s = c->scratch;
  c->status = reinterpret_cast<int*>(s + c->sl.status);
  c->counters = reinterpret_cast<int*>(s + c->sl.counters);
  c->prompt = reinterpret_cast<int32_t*>(s + c->sl.prompt);
  c->slot_len = reinterpret_cast<int*>(s + c->sl.slot_len);
  c->match_out = reinterpret_cast<int32_t*>(s + c->sl.match_out);
  c->rope = reinterpret_cast<float2*>(s + c->sl.rope);
  c->rope_fr = rope_freq(cfg->rope_theta, cfg->head_dim);
  c->h = reinterpret_cast<float*>(s + c->sl.h);
  c->a = reinterpret_cast<__nv_bfloat16*>(s + c->sl.a);
  c->q = reinterpret_cast<__nv_bfloat16*>(s + c->sl.q);
  c->o = reinterpret_cast<__nv_bfloat16*>(s + c->sl.o);
  c->z = reinterpret_cast<__nv_bfloat16*>(s + c->sl.z);
  c->part = reinterpret_cast<float*>(s + c->sl.part);
  c->opart = reinterpret_cast<float*>(s + c->sl.opart);
  c->ml = reinterpret_cast<float2*>(s + c->sl.ml);
  c->best = reinterpret_cast<float2*>(s + c->sl.best);
  c->next = reinterpret_cast<int32_t*>(s + c->sl.next);
  c->pass_layers = reinterpret_cast<PassLayer*>(s + c->sl.pass_layers);
  c->pass_done = reinterpret_cast<int*>(s + c->sl.pass_done);
  c->pass_ss = reinterpret_cast<float*>(s + c->sl.pass_ss);
  c->pass_diag = reinterpret_cast<int*>(s + c->sl.pass_diag);

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->n_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = gemv_setup();
  if (e == cudaSuccess) e = gemm_tc_setup();
  if (e == cudaSuccess) e = attn_setup();
  if (e == cudaSuccess) e = attn_tc_setup();
  // the persistent pass is optional: without room for it, small m keeps the
  // per-step launches
  if (e == cudaSuccess && pass_setup() != cudaSuccess) {
    (void)cudaGetLastError();
    c->use_pass = false;
  }
  if (e == cudaSuccess && !g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess) g_encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    else if (e == cudaSuccess) e = cudaErrorNotSupported;
  }
  if (e != cudaSuccess) {
    delete c;
    return KVR_ERR_CUDA;
  }
  const kvr_config& k = *cfg;
  const uint64_t kv_rows = (uint64_t)c->granted * k.n_layers * 2 * k.n_kv_heads * k.capacity;
  bool ok = encode_2d(&c->tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->arena, k.head_dim, kv_rows,
                      (uint64_t)k.head_dim * 2, 64, kAttnKeys, CU_TENSOR_MAP_SWIZZLE_128B);
  // the same arena as [rows][capacity]: V^T tiles of head_dim rows x 64 keys
  ok = ok && encode_2d(&c->tm_vt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->arena, k.capacity,
                       kv_rows * k.head_dim / k.capacity, (uint64_t)k.capacity * 2, 64, k.head_dim,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && encode_2d(&c->tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c->q, k.head_dim,
                       (uint64_t)k.max_rows * k.n_q_heads, (uint64_t)k.head_dim * 2, 64, 128,
                       CU_TENSOR_MAP_SWIZZLE_128B);
  if (packed4(k)) {
    ok = ok && act_maps(c->tm_a, c->a, k.hidden, k.max_rows);
    ok = ok && act_maps(c->tm_o, c->o, k.n_q_heads * k.head_dim, k.max_rows);
    if (!k.attn_only) ok = ok && act_maps(c->tm_z, c->z, k.ffn, k.max_rows);
  }
  if (!ok) {
    delete c;
    return KVR_ERR_CUDA;
  }
  // Positions past a slot's length are read (and multiplied by a zero weight)
  // when a key block is partly visible; zero the arena once so they are finite.
  e = cudaMemset(c->status, 0, 64);
  if (e == cudaSuccess) e = cudaMemset(c->counters, 0, (kCounters + kAttnCounters) * 4);
  if (e == cudaSuccess) e = cudaMemset(c->pass_done, 0, ((size_t)k.n_layers * kPassPhases + 8) * 4);
  if (e == cudaSuccess) e = cudaMemset(c->pass_diag, 0, (size_t)kPassMaxCtas * 2 * 4);
  if (e == cudaSuccess && cudaHostAlloc(&c->pass_host, (size_t)k.n_layers * sizeof(PassLayer), cudaHostAllocDefault) != cudaSuccess) {
    (void)cudaGetLastError();
    c->pass_host = nullptr;
    c->use_pass = false;
  }
  if (e == cudaSuccess) e = cudaMemset(c->arena, 0, (size_t)c->granted * slot_kv_bytes(cfg));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    delete c;
    return KVR_ERR_CUDA;
  }
  c->host_match_n = (size_t)(c->granted + 1) * c->granted;
  if (cudaHostAlloc(&c->host_match, c->host_match_n * 4, cudaHostAllocDefault) != cudaSuccess) {
    delete c;
    return KVR_ERR_CUDA;
  }
  *out = c;
  return KVR_OK;
}

int kvr_ctx_info(const kvr_ctx* c, int* slots_granted, int* slots_requested, int* capacity) {
  if (!c) return KVR_ERR_ARG;
  if (slots_granted) *slots_granted = c->granted;
  if (slots_requested) *slots_requested = c->requested;
  if (capacity) *capacity = c->cfg.capacity;
  return KVR_OK;
}

int kvr_ctx_destroy(kvr_ctx* c) {
  if (!c) return KVR_ERR_ARG;
  for (auto& p : c->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : c->free_events) cudaEventDestroy(e);
  if (c->host_match) cudaFreeHost(c->host_match);
  if (c->pass_host) cudaFreeHost(c->pass_host);
  delete c;
  return KVR_OK;
}

int kvr_slot_match(kvr_ctx* c, const int32_t* tokens, int n, int* slot, int* reused, void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (!tokens || !slot || !reused || n <= 0) return fail(c, KVR_ERR_ARG, "null pointer or n <= 0");
  if (n > c->cfg.capacity) return fail(c, KVR_ERR_CAPACITY, "prompt of %d tokens exceeds capacity %d", n, c->cfg.capacity);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int S = c->granted;
  if (!c->reuse) {
    match_without_reuse(c, slot, reused);
    return KVR_OK;
  }
  int lens[KVR_MAX_SLOTS];
  for (int s = 0; s < S; ++s) lens[s] = c->slots[s].occupied ? (int)c->slots[s].tokens.size() : -1;
  cudaError_t e = cudaMemcpyAsync(c->prompt, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->slot_len, lens, (size_t)S * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(c, e, "match upload");
  {
    Timed t(c, kMatch, st);
    e = launch_prefix_match(c->tok_mirror, c->slot_len, S, c->cfg.capacity, c->prompt, n,
                            c->match_out, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "prefix match launch");
  e = cudaMemcpyAsync(c->host_match, c->match_out, c->host_match_n * 4,
                      cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(c, e, "match readback");
  apply_slot_policy(c, c->host_match, n, slot, reused);
  return KVR_OK;
}

int kvr_slot_truncate(kvr_ctx* c, int slot, int new_len) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slot);
  const int len = (int)c->slots[slot].tokens.size();
  if (new_len < 0 || new_len > len) return fail(c, KVR_ERR_ARG, "truncate to %d outside [0, %d]", new_len, len);
  c->slots[slot].tokens.resize(new_len);
  return KVR_OK;
}

int kvr_slot_len(const kvr_ctx* c, int slot, int* len) {
  if (!c || !len || slot < 0 || slot >= c->granted) return KVR_ERR_ARG;
  *len = (int)c->slots[slot].tokens.size();
  return KVR_OK;
}

int kvr_slot_tokens(const kvr_ctx* c, int slot, int32_t* tokens, int n) {
  if (!c || !tokens || n < 0 || slot < 0 || slot >= c->granted) return KVR_ERR_ARG;
  const int k = std::min(n, (int)c->slots[slot].tokens.size());
  if (k > 0) memcpy(tokens, c->slots[slot].tokens.data(), (size_t)k * 4);
  return KVR_OK;
}

int kvr_slot_assign(kvr_ctx* c, int slot, const int32_t* tokens, int n, void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slot);
  if (n < 0 || (n > 0 && !tokens)) return fail(c, KVR_ERR_ARG, "bad token list");
  if (n > c->cfg.capacity) return fail(c, KVR_ERR_CAPACITY, "%d tokens exceed capacity %d", n, c->cfg.capacity);
  int rc = upload_tokens(c, slot, 0, tokens, n, static_cast<cudaStream_t>(stream));
  if (rc) return rc;
  c->slots[slot].occupied = true;
  c->slots[slot].tokens.assign(tokens, tokens + n);
  touch(c, slot);
  return KVR_OK;
}

uint64_t kvr_config_hash(const kvr_config* cfg, uint64_t model_tag) {
  if (!cfg) return 0;
  const uint32_t w[10] = {(uint32_t)cfg->n_layers,      (uint32_t)cfg->hidden,   (uint32_t)cfg->n_q_heads,
                          (uint32_t)cfg->n_kv_heads,    (uint32_t)cfg->head_dim, (uint32_t)cfg->ffn,
                          (uint32_t)cfg->weight_format, (uint32_t)cfg->attn_only, float_word(cfg->rope_theta),
                          float_word(cfg->rms_eps)};
  return fnv1a_words(w, 10, model_tag);
}

size_t kvr_slot_spill_bytes(const kvr_ctx* c, int slot) {
  if (!c || slot < 0 || slot >= c->granted) return 0;
  return spill_layout((int)c->slots[slot].tokens.size(), c->cfg.n_layers, c->cfg.n_kv_heads, c->cfg.head_dim).total;
}

int kvr_slot_spill(kvr_ctx* c, int slot, uint64_t model_tag, void* host, size_t bytes, void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted || !host) return fail(c, KVR_ERR_ARG, "bad slot %d or null record", slot);
  const kvr_config& k = c->cfg;
  const int len = (int)c->slots[slot].tokens.size();
  const SpillLayout L = spill_layout(len, k.n_layers, k.n_kv_heads, k.head_dim);
  if (bytes < L.total) return fail(c, KVR_ERR_CAPACITY, "spill of slot %d needs %zu bytes", slot, L.total);
  uint8_t* rec = static_cast<uint8_t*>(host);
  SpillHeader hd;
  memset(&hd, 0, sizeof hd);
  memcpy(hd.magic, kSpillMagic, 8);
  hd.hash = kvr_config_hash(&k, model_tag);
  hd.bytes = L.total;
  hd.len = len;
  hd.n_layers = k.n_layers;
  hd.n_kv_heads = k.n_kv_heads;
  hd.head_dim = k.head_dim;
  memcpy(rec, &hd, sizeof hd);
  memset(rec + L.tokens, 0, L.kv - L.tokens);
  if (len > 0) memcpy(rec + L.tokens, c->slots[slot].tokens.data(), (size_t)len * 4);
  cudaError_t e = copy_slot_kv(c, slot, len, rec, true, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVR_OK : cuda_fail(c, e, "slot spill copy");
}

int kvr_slot_restore(kvr_ctx* c, int slot, uint64_t model_tag, const void* host, size_t bytes, void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted || !host) return fail(c, KVR_ERR_ARG, "bad slot %d or null record", slot);
  const kvr_config& k = c->cfg;
  if (bytes < sizeof(SpillHeader)) return fail(c, KVR_ERR_ARG, "record shorter than its header");
  SpillHeader hd;
  memcpy(&hd, host, sizeof hd);
  if (memcmp(hd.magic, kSpillMagic, 8)) return fail(c, KVR_ERR_ARG, "not a slot record");
  if (hd.hash != kvr_config_hash(&k, model_tag))
    return fail(c, KVR_ERR_MISMATCH, "slot record from another model or KV layout");
  if (hd.n_layers != k.n_layers || hd.n_kv_heads != k.n_kv_heads || hd.head_dim != k.head_dim || hd.len < 0)
    return fail(c, KVR_ERR_ARG, "damaged slot record header");
  const SpillLayout L = spill_layout(hd.len, k.n_layers, k.n_kv_heads, k.head_dim);
  if (hd.bytes != L.total || bytes < L.total) return fail(c, KVR_ERR_ARG, "slot record truncated or damaged");
  if (hd.len > k.capacity) return fail(c, KVR_ERR_CAPACITY, "record of %d tokens exceeds capacity %d", hd.len, k.capacity);
  const uint8_t* rec = static_cast<const uint8_t*>(host);
  const int32_t* toks = reinterpret_cast<const int32_t*>(rec + L.tokens);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SlotState& S = c->slots[slot];
  cudaError_t e = copy_slot_kv(c, slot, hd.len, const_cast<uint8_t*>(rec), false, st);
  int rc = e == cudaSuccess ? upload_tokens(c, slot, 0, toks, hd.len, st) : cuda_fail(c, e, "slot restore copy");
  if (rc) {   // the slot's K/V may be partly overwritten: leave it empty
    S.tokens.clear();
    return rc;
  }
  S.occupied = true;
  S.tokens.assign(toks, toks + hd.len);
  touch(c, slot);
  return KVR_OK;
}

int kvr_slot_kv(const kvr_ctx* c, int slot, int layer, void** k, void** v) {
  if (!c || slot < 0 || slot >= c->granted || layer < 0 || layer >= c->cfg.n_layers) return KVR_ERR_ARG;
  __nv_bfloat16* base = reinterpret_cast<__nv_bfloat16*>(c->arena);
  if (k) *k = base + kv_offset(c, slot, layer, 0);
  if (v) *v = base + kv_offset(c, slot, layer, 1);
  return KVR_OK;
}

int kvr_prefill_suffix(kvr_ctx* c, int slot, const int32_t* tokens, int m, const void* hidden,
                       const kvr_layer_weights* w, void* out, void* stream) {
  return prefill_common(c, slot, tokens, m, hidden, w, out, stream, 1 << 30);
}

int kvr_verify(kvr_ctx* c, int slot, const int32_t* tokens, int m, const void* hidden,
               const kvr_layer_weights* w, void* out, void* stream) {
  return prefill_common(c, slot, tokens, m, hidden, w, out, stream, kVerifyMaxRows);
}

int kvr_verify_accept(kvr_ctx* c, int slot, const int32_t* tokens, int m, const void* hidden,
                      const kvr_layer_weights* w, const kvr_head_weights* head, void* out,
                      int32_t* next_tokens, int* accepted, void* stream) {
  if (!c) return KVR_ERR_ARG;
  int rc = head_check(c, head, next_tokens, accepted);
  if (rc) return rc;
  if (slot < 0 || slot >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slot);
  const int p0 = (int)c->slots[slot].tokens.size();
  rc = prefill_common(c, slot, tokens, m, hidden, w, out, stream, kVerifyMaxRows,
                      static_cast<const __nv_bfloat16*>(head->norm));
  if (rc) return rc;
  rc = head_decide(c, static_cast<cudaStream_t>(stream), m, head, next_tokens);
  if (rc) {
    c->slots[slot].tokens.resize(p0);
    return rc;
  }
  const int a = greedy_accept(tokens, next_tokens, m);
  *accepted = a;
  c->slots[slot].tokens.resize(p0 + 1 + a);
  return KVR_OK;
}

int kvr_prefill_branches(kvr_ctx* c, int slot, int n_branch, const int* lens, const int32_t* tokens,
                         const void* hidden, const kvr_layer_weights* w, void* out, void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (slot < 0 || slot >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slot);
  if (n_branch < 1 || n_branch > KVR_MAX_BRANCHES || !lens || !tokens || !hidden || !out)
    return fail(c, KVR_ERR_ARG, "bad branch arguments");
  if (((uintptr_t)hidden & 15) || ((uintptr_t)out & 15)) return fail(c, KVR_ERR_ARG, "hidden/out must be 16-byte aligned");
  if (!weights_ok(c, w)) return fail(c, KVR_ERR_ARG, "missing or misaligned weight pointer");
  RowMap rows;
  memset(&rows, 0, sizeof rows);
  rows.P = (int)c->slots[slot].tokens.size();
  rows.n_branch = n_branch;
  rows.slot[0] = slot;
  int total = 0;
  for (int b = 0; b < n_branch; ++b) {
    if (lens[b] <= 0) return fail(c, KVR_ERR_ARG, "branch %d has %d rows", b, lens[b]);
    rows.off[b] = total;
    total += lens[b];
  }
  rows.off[n_branch] = total;
  rows.m = total;
  if (total > c->cfg.max_rows || rows.P + total > c->cfg.capacity || c->fault == 3)
    return fail(c, KVR_ERR_CAPACITY, "%d branch rows after %d exceed capacity %d (max_rows %d)", total,
                rows.P, c->cfg.capacity, c->cfg.max_rows);
  if (c->fault == 2) return fail(c, KVR_ERR_FAULT, "injected launch fault");
  int rc = run_stack(c, rows, hidden, w, out, static_cast<cudaStream_t>(stream));
  if (rc) return rc;
  c->slots[slot].occupied = true;
  touch(c, slot);
  return KVR_OK;
}

int kvr_prefill_batch(kvr_ctx* c, int n_seq, const int* slots, const int* lens, const int32_t* tokens,
                      const void* hidden, const kvr_layer_weights* w, void* out, void* stream) {
  return batch_common(c, n_seq, slots, lens, tokens, hidden, w, out, stream, 1 << 30, nullptr);
}

int kvr_verify_accept_batch(kvr_ctx* c, int n_seq, const int* slots, const int* lens, const int32_t* tokens,
                            const void* hidden, const kvr_layer_weights* w, const kvr_head_weights* head,
                            void* out, int32_t* next_tokens, int* accepted, void* stream) {
  if (!c) return KVR_ERR_ARG;
  int rc = head_check(c, head, next_tokens, accepted);
  if (rc) return rc;
  if (n_seq < 1 || n_seq > KVR_MAX_BRANCHES || !slots || !lens) return fail(c, KVR_ERR_ARG, "bad batch arguments");
  int p0[KVR_MAX_BRANCHES];
  for (int j = 0; j < n_seq; ++j) {
    if (slots[j] < 0 || slots[j] >= c->granted) return fail(c, KVR_ERR_ARG, "bad slot %d", slots[j]);
    p0[j] = (int)c->slots[slots[j]].tokens.size();
  }
  rc = batch_common(c, n_seq, slots, lens, tokens, hidden, w, out, stream, kVerifyMaxRows,
                    static_cast<const __nv_bfloat16*>(head->norm));
  if (rc) return rc;
  int total = 0;
  for (int j = 0; j < n_seq; ++j) total += lens[j];
  rc = head_decide(c, static_cast<cudaStream_t>(stream), total, head, next_tokens);
  if (rc) {
    for (int j = 0; j < n_seq; ++j) c->slots[slots[j]].tokens.resize(p0[j]);
    return rc;
  }
  int at = 0;
  for (int j = 0; j < n_seq; ++j) {
    accepted[j] = greedy_accept(tokens + at, next_tokens + at, lens[j]);
    c->slots[slots[j]].tokens.resize(p0[j] + 1 + accepted[j]);
    at += lens[j];
  }
  return KVR_OK;
}

int kvr_sync_status(kvr_ctx* c, void* stream) {
  if (!c) return KVR_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int word = 0;
  cudaError_t e = cudaMemcpyAsync(&word, c->status, 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(c, e, "status readback");
  if (word) {
    // where the small-m pass's waits gave up, if it ran: (site, detail, CTA)
    // of the first few CTAs that recorded one
    std::string where;
    std::vector<int> diag((size_t)kPassMaxCtas * 2);
    e = cudaMemcpyAsync(diag.data(), c->pass_diag, diag.size() * 4, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(c, e, "status detail readback");
    int shown = 0, total = 0;
    for (int b = 0; b < kPassMaxCtas; ++b) {
      const int code = diag[2 * b];
      if (!code) continue;
      ++total;
      if (shown < 6) {
        char buf[96];
        snprintf(buf, sizeof buf, "%s[cta %d site %d detail %d seen %d]", shown ? " " : "; pass waits: ",
                 (code >> 16) & 0x7FFF, (code >> 1) & 7, (code >> 4) & 0xFFF, diag[2 * b + 1]);
        where += buf;
        ++shown;
      }
    }
    if (total > shown) where += " ... (" + std::to_string(total) + " CTAs)";
    // a launch that gave up may have left arrival counters behind: clear
    // every one of them (GEMV tiles and split-KV merges) and the status word
    e = cudaMemsetAsync(c->counters, 0, (kCounters + kAttnCounters) * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(c->pass_diag, 0, (size_t)kPassMaxCtas * 2 * 4, st);
    if (e == cudaSuccess)
      e = cudaMemsetAsync(c->pass_done, 0, ((size_t)c->cfg.n_layers * kPassPhases + 8) * 4, st);
    c->pass_epoch = 0;
    if (e == cudaSuccess) e = cudaMemsetAsync(c->status, 0, 4, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(c, e, "clearing the counters after a timeout");
    return fail(c, KVR_ERR_TIMEOUT, "a device-side wait gave up (status %d)%s", word, where.c_str());
  }
  return KVR_OK;
}

int kvr_selftest_wait(kvr_ctx* c, void* stream) {
  if (!c) return KVR_ERR_ARG;
  cudaError_t e = launch_wait_probe(c->status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVR_OK : cuda_fail(c, e, "wait probe launch");
}

int kvr_trace_set(kvr_ctx* c, void* dev, size_t bytes) {
  if (!c) return KVR_ERR_ARG;
  if (!dev) {
    c->trace = nullptr;
    return KVR_OK;
  }
  const size_t need = (size_t)(c->cfg.n_layers + 1) * c->cfg.max_rows * c->cfg.hidden * 4;
  if (bytes < need) return fail(c, KVR_ERR_CAPACITY, "trace buffer needs %zu bytes", need);
  if ((uintptr_t)dev & 15) return fail(c, KVR_ERR_ARG, "trace buffer must be 16-byte aligned");
  c->trace = static_cast<float*>(dev);
  return KVR_OK;
}

int kvr_profile_enable(kvr_ctx* c, int on) {
  if (!c) return KVR_ERR_ARG;
  c->prof = on != 0;
  return KVR_OK;
}

int kvr_profile_launches(kvr_ctx* c, int* cls, float* ms, int max_n, int* n) {
  if (!c || !n || max_n < 0 || (max_n > 0 && (!cls || !ms))) return KVR_ERR_ARG;
  int k = 0;
  for (auto& p : c->pending) {
    cudaError_t e = cudaEventSynchronize(p.b);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, p.a, p.b);
    if (e != cudaSuccess) return cuda_fail(c, e, "profile events");
    if (k < max_n) {
      cls[k] = p.cls;
      ms[k] = t;
    }
    ++k;
  }
  *n = k;
  return KVR_OK;
}

int kvr_profile_read(kvr_ctx* c, float ms[4], int launches[4]) {
  if (!c) return KVR_ERR_ARG;
  for (auto& p : c->pending) {
    cudaError_t e = cudaEventSynchronize(p.b);
    float t = 0.f;
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, p.a, p.b);
    if (e == cudaSuccess) c->prof_ms[p.cls] += t;
    c->free_events.push_back(p.a);
    c->free_events.push_back(p.b);
  }
  c->pending.clear();
  for (int i = 0; i < 4; ++i) {
    if (ms) ms[i] = c->prof_ms[i];
    if (launches) launches[i] = c->prof_launches[i];
    c->prof_ms[i] = 0.f;
    c->prof_launches[i] = 0;
  }
  return KVR_OK;
}

const char* kvr_last_error(const kvr_ctx* c) { return c ? c->err.c_str() : "null context"; }

// kvr_slot_match with its device staging in the library's static array
// (k_match_static.cu) instead of the context's scratch area; the policy applied
// to the match lengths is the one of kvr_slot_match.
int kvr_slot_match_static(kvr_ctx* c, const int32_t* tokens, int n, int* slot, int* reused,
                          void* stream) {
  if (!c) return KVR_ERR_ARG;
  if (!tokens || !slot || !reused || n <= 0) return fail(c, KVR_ERR_ARG, "null pointer or n <= 0");
  if (n > KVR_STATIC_MATCH_MAX_TOKENS)
    return fail(c, KVR_ERR_CAPACITY, "prompt of %d tokens exceeds the static match limit of %d tokens",
                n, KVR_STATIC_MATCH_MAX_TOKENS);
  if (n > c->cfg.capacity) return fail(c, KVR_ERR_CAPACITY, "prompt of %d tokens exceeds capacity %d", n, c->cfg.capacity);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int S = c->granted;
  if (!c->reuse) {
    match_without_reuse(c, slot, reused);
    return KVR_OK;
  }
  int32_t *d_prompt = nullptr, *d_out = nullptr;
  int* d_len = nullptr;
  cudaError_t e = static_match_scratch(&d_prompt, &d_len, &d_out);
  if (e != cudaSuccess) return cuda_fail(c, e, "static match scratch lookup");
  int lens[KVR_MAX_SLOTS];
  for (int s = 0; s < S; ++s) lens[s] = c->slots[s].occupied ? (int)c->slots[s].tokens.size() : -1;
  e = cudaMemcpyAsync(d_prompt, tokens, (size_t)n * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_len, lens, (size_t)S * 4, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(c, e, "static match upload");
  {
    Timed t(c, kMatch, st);
    e = launch_prefix_match(c->tok_mirror, d_len, S, c->cfg.capacity, d_prompt, n, d_out, st);
  }
  if (e != cudaSuccess) return cuda_fail(c, e, "prefix match launch");
  std::vector<int32_t> res((size_t)(S + 1) * S);
  e = cudaMemcpyAsync(res.data(), d_out, res.size() * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(c, e, "static match readback");
  apply_slot_policy(c, res.data(), n, slot, reused);
  return KVR_OK;
}

}  // extern "C"
