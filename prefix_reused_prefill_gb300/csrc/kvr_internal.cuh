// Internal declarations shared by the kvr kernels and the C-ABI host code.
// sm_103a only: TMA (cp.async.bulk.tensor), mbarrier transaction counts,
// ldmatrix and bf16 tensor-core fragments are used directly through inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvr.h"

namespace kvr {

// ----------------------------------------------------------------------------
// constants
// ----------------------------------------------------------------------------
constexpr int kGemvRows = 128;     // weight rows per GEMV CTA (8 warps x 16 rows)
constexpr int kGemvKStep = 256;    // inputs per pipeline stage (8 groups of 32)
constexpr int kGemvMaxCols = 32;   // tokens per GEMV pass (4 tensor-core n-tiles)
constexpr int kMaxKSplit = 16;
constexpr int kGemmMaxTok = 256;   // tokens per tcgen05 GEMM pass (MMA N <= 256)
constexpr int kGemmMaxSplit = 8;
constexpr int kAttnKeys = 64;      // keys per attention pipeline stage
constexpr int kAttnTcMinRows = 96; // G*m above this: tcgen05 attention (128-row tiles)
constexpr int kAttnTcKeys = 128;   // keys per block of the tcgen05 attention
constexpr int kSplitTargetCtas = 320;
constexpr int kMaxSplits = 64;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // 1 s per bounded wait

constexpr int kStatusTimeout = 1;

// Rows of one call: P committed keys visible to every row; row i of branch b
// (off[b] <= i < off[b+1]) sits at position P + i - off[b], is stored at slot
// index P + i, and also sees slot indices [P + off[b], P + i].
// The m rows of one call, in branches b = rows [off[b], off[b+1]):
//  * batch == 0 (one slot, slot[0]): keys [0, P) are the shared cached prefix;
//    row i is stored at P + i and sits at position P + i - off[b]; it sees
//    the prefix and its own branch's rows up to itself (a plain suffix is the
//    one-branch case).
//  * batch == 1 (one conversation per branch): branch b appends to slot[b]
//    after that slot's pre[b] cached tokens, exactly as a one-branch call on
//    that slot would (row i at position and index pre[b] + i - off[b]).
struct RowMap {
  int P;
  int m;
  int n_branch;
  int batch;
  int off[KVR_MAX_BRANCHES + 1];
  int pre[KVR_MAX_BRANCHES];
  int slot[KVR_MAX_BRANCHES];
};

__host__ __device__ inline int row_branch(const RowMap& r, int i) {
  int b = 0;
  while (b + 1 < r.n_branch && i >= r.off[b + 1]) ++b;
  return b;
}

// RoPE position of row i
__host__ __device__ inline int row_pos(const RowMap& r, int i) {
  const int b = row_branch(r, i);
  return (r.batch ? r.pre[b] : r.P) + i - r.off[b];
}

// slot and slot index receiving row i's K/V
__host__ __device__ inline int row_slot(const RowMap& r, int i) { return r.slot[r.batch ? row_branch(r, i) : 0]; }
__host__ __device__ inline int row_store(const RowMap& r, int i) {
  if (!r.batch) return r.P + i;
  const int b = row_branch(r, i);
  return r.pre[b] + i - r.off[b];
}

// q buffer row ([rows][head_dim]) of row i, query head g of KV head kv:
// KV-head-major [Hkv][m][G] per call, or per conversation in a batch (the
// block of branch b starts at row off[b] * Hq) so each conversation's
// attention reads a [Hkv][len][G] block of its own
__host__ __device__ inline long long q_row(const RowMap& r, int i, int kv, int g, int G, int Hq) {
  if (!r.batch) return ((long long)kv * r.m + i) * G + g;
  const int b = row_branch(r, i);
  const int len = r.off[b + 1] - r.off[b];
  return (long long)r.off[b] * Hq + ((long long)kv * len + (i - r.off[b])) * G + g;
}

// ----------------------------------------------------------------------------
// kernel parameter blocks
// ----------------------------------------------------------------------------
struct GemvSeg {
  CUtensorMap tw;   // int4: uint8 [N][K/2], box {128 B, 128 rows}, 128B swizzle
  CUtensorMap ts;   // int4: fp16 scales [N][K/32], box {8, 128 rows}
  const __nv_bfloat16* wbf;  // bf16 weights [N][K] (bf16 format only)
  int N;
  int col0;         // first output column of this segment
  int tile0;        // first CTA tile of this segment
  int tiles;
};

// Epilogue the int4 GEMV applies itself (the last CTA of a tile to finish
// adds the k-split partials in split order and then):
enum GemvEpi : int {
  kGemvEpiQKV = 0,     // RoPE q and k, round to bf16, write q, append K and V^T to the slot
  kGemvEpiResid = 1,   // h += y (fp32 residual stream); optionally out = bf16(h)
  kGemvEpiSwiglu = 2,  // tile = 64 gate rows + the same 64 up rows: z = bf16(silu(g) * u)
  kGemvEpiCast = 3,    // out = bf16(y)
  kGemvEpiArgmax = 4,  // per token, the tile's largest y and its row (lowest on ties) -> best
};

// int4 weight formats of the GEMV and the tcgen05 GEMM (include/kvr.h):
// group-32 fp16 scales, or K-quant superblocks (16-byte records per 256 inputs)
enum WeightFmt { kFmtInt4 = 0, kFmtQ4K = 1 };

struct GemvParams {
  GemvSeg seg[3];   // SwiGLU: seg[0] = gate, seg[1] = up (64-row boxes), nseg = 1
  CUtensorMap tx;   // activations bf16 [max_rows][K], box {64, 8*NT}, 128B swizzle
  const __nv_bfloat16* x;  // same activations, plain pointer (bf16 kernel)
  int nseg;
  int K;
  int ksteps;       // 256-input steps along K
  int ksplit;       // bf16 kernel only (always 1)
  int ctas;         // int4 kernel: CTA i takes units [i*U/ctas, (i+1)*U/ctas), U = tiles*ksteps
  int maxc;         // int4 kernel: partial slots per tile (>= contributors of any tile)
  int c0;           // first token of this pass
  int mb;           // tokens in this pass (<= kGemvMaxCols)
  int ldo;          // partial row stride (total output columns; bf16 kernel)
  long long plane;  // floats per split plane of the partials (bf16 kernel)
  float* part;      // bf16 kernel: [kGemvMaxCols][ldo]; int4 kernel: [tiles][maxc][32][128]
  int* status;
  // fused epilogue of the int4 kernel
  int epi;          // GemvEpi
  int fmt;          // WeightFmt
  int tiles;        // tiles of this launch
  int* counters;    // [tiles] contributor arrival counters; zero between launches
  RowMap rows;      // QKV: row positions (row i is stored at rows.P + i)
  const float2* rope;   // QKV: (cos, sin) [m][d/2]
  __nv_bfloat16* q;     // QKV: [Hkv][m][G][d]
  __nv_bfloat16* arena; // QKV: the slot arena
  long long k_off, v_off;   // QKV: the layer's K and V^T in slot 0
  long long slot_stride;    // QKV: arena elements per slot
  int cap, Hq, Hkv, d;
  float* h;             // Resid: [max_rows][H]
  int H;
  __nv_bfloat16* out;   // Resid (last layer) / Cast: bf16 [m][ldout], or null
  int ldout;
  __nv_bfloat16* z;     // Swiglu: [max_rows][F]
  int F;
  float2* best;         // Argmax: [token][tiles] (value, row)
};

struct GemmSeg {
  CUtensorMap tw;        // uint8 [N][K/2], box {64 B, 128 rows} (64 rows for SwiGLU), 64B swizzle
  const __half* scales;  // fp16 [N][K/32]
  int N;
  int col0;
  int tile0;
  int tiles;
};

struct GemmParams {
  GemmSeg seg[3];   // SwiGLU mode: seg[0] = gate, seg[1] = up (nseg = 1 for tiling)
  CUtensorMap tx;   // activations bf16 [max_rows][K], box {64, xrows}, 128B swizzle
  int nseg;
  int K;
  int kchunks;      // K / 128 (pipeline stages)
  int ksplit;
  int n_tok;        // MMA N: tokens of this pass rounded up to 16 (<= 256)
  int xrows;        // activation box rows (64, 128 or 256) >= n_tok
  int m;            // valid tokens of this pass
  int t0;           // first token of this pass
  int swiglu;       // 1: write z = silu(gate) * up; 0: write fp32 partial sums
  int fmt;          // WeightFmt (scales: fp16 group scales or K-quant records)
  int exact;        // weights as two fp16 terms (hi + lo, two MMAs): exact code * scale
  int ldo;
  int F;
  long long plane;
  float* part;      // [ksplit][256][ldo]
  __nv_bfloat16* z; // [max_rows][F]
  int z16;          // z holds fp16 (the next GEMM's operand type)
  int* status;
};

// One conversation of a batched small-m attention launch.
struct AttnConv {
  int kbase, vtbase;   // its slot's K / V^T rows of the layer (as AttnParams)
  int P, m;            // its cached tokens and new rows
  int tok0;            // its first row in the call
  int tile0;           // its first row tile (blockIdx.x)
  int nsplit;
  long long part0;     // float offset of its partials [nsplit][m][Hq][d] (ml: part0 / d)
};

struct AttnParams {
  CUtensorMap tkv;           // arena as bf16 [rows][head_dim], box {64, 64}, 128B swizzle (K tiles)
  CUtensorMap tvt;           // arena as bf16 [rows][capacity], box {64, head_dim} (V^T tiles)
  CUtensorMap tq;            // q as bf16 [Hkv*max_rows*G][head_dim], box {64, 128}
  const __nv_bfloat16* q;    // [Hkv][m][G][d] after RoPE (KV-head-major rows)
  __nv_bfloat16* o;          // [m][Hq*d] (nsplit == 1)
  float* opart;              // [nsplit][m][Hq][d]
  float2* ml;                // [nsplit][m][Hq]  (running max in log2 units, sum)
  RowMap rows;
  int Hq, Hkv, G;
  int qrow0;                 // first q buffer row of this launch (a conversation of a batch)
  int kbase;                 // [rows][d] view row of (slot, layer, K, head 0, position 0)
  int vtbase;                // [rows][cap] view row of (slot, layer, V^T, head 0, element 0)
  int cap;
  int nsplit;
  int row_tiles;
  float scale_log2;          // log2(e) / sqrt(d)
  int o16;                   // o holds fp16 (the O projection runs on the tcgen05 GEMM)
  int* status;
  // split-KV kernel with one row tile (R <= 16): arrival counters per (row
  // tile, KV head), zero between launches; the last split merges the splits
  // and writes o itself (no combine launch).  Null: the combine kernel merges.
  int* counters;
  // batched conversations (split-KV kernel and combine only): n_conv > 0
  // replaces rows/kbase/vtbase/nsplit/q/o by each CTA's conversation
  int n_conv;
  AttnConv conv[KVR_MAX_BRANCHES];
};

// Persistent small-m pass: the whole stack for up to kPassRows rows in one
// cooperative launch (k_pass.cu).
constexpr int kPassRows = 16;       // rows of a call (two tensor-core n-tiles)
constexpr int kPassMaxAttnRows = 64;   // G * rows: four 16-row attention tiles
constexpr int kPassPhases = 5;      // QKV, attention, O, gate|up, down per layer
constexpr int kPassMaxCtas = 512;   // per-CTA records of a wait that gave up

// per-layer weight descriptors, in device memory (tensor maps 64-byte aligned)
struct PassLayer {
  CUtensorMap tw[7];   // int4 bytes of wq wk wv wo wg wu wd: 128-row boxes (wg, wu: 64-row boxes)
  CUtensorMap ts[7];   // their fp16 scales, same row boxes
  const __nv_bfloat16* norm_attn;
  const __nv_bfloat16* norm_ffn;
};
static_assert(alignof(PassLayer) >= 64 && sizeof(PassLayer) % 64 == 0,
              "every layer's tensor maps stay 64-byte aligned in the device table");

struct PassParams {
  const PassLayer* layers;
  int L, H, F, Hq, Hkv, d, G, cap;
  int m;                   // rows of the call
  RowMap rows;             // one slot (batch == 0); branches allowed
  int slot;
  CUtensorMap tkv, tvt;    // the arena as the attention kernels see it
  __nv_bfloat16* arena;
  long long kv_slot;       // arena elements before (slot, layer 0, K)
  int kbase0, vtbase0;     // [rows][d] / [rows][cap] view rows of (slot, layer 0)
  int ctas;
  int maxc[kPassPhases];   // partial slots per tile of each projection phase
  int nsplit, nb;          // attention: key splits per KV head, 64-key blocks over [0, P + m)
  const __nv_bfloat16* hidden;
  float* h;                // [m][H] residual stream
  float* ss;               // [m][nss] sum of h^2 per 128-column tile
  int nss;
  const float2* rope;      // (cos, sin) [m][d/2]
  __nv_bfloat16* q;        // [Hkv][m][G][d]
  __nv_bfloat16* o;        // [m][Hq*d]
  __nv_bfloat16* z;        // [m][F]
  float* part;             // projection partials [tiles][maxc][32][128]
  float* opart;            // attention partials [Hkv*nsplit][64][d]
  float2* ml;              // [Hkv*nsplit][64] (max in log2 units, sum)
  int* tile_cnt;           // per-tile arrivals (zero between uses)
  int* head_cnt;           // per-KV-head split arrivals (zero between uses)
  int* done;               // [L*5 + 1] completion counters, growing by one call's count per call
  unsigned epoch;          // this call: a counter is complete at epoch * its count
  __nv_bfloat16* out;      // bf16 [m][H] (last layer), or null
  const __nv_bfloat16* head_gain;  // output head's RMSNorm: a_head = bf16(RMSNorm(h) * gain), or null
  __nv_bfloat16* a_head;
  float* trace;            // [L + 1][trace_rows][H] layer inputs (float32), or null
  int trace_rows;
  int* diag;               // [kPassMaxCtas][2]: a CTA's wait that gave up (code, value seen)
  float eps, scale_log2;
  int* status;
};

// ----------------------------------------------------------------------------
// launchers (each returns the error of its launch)
// ----------------------------------------------------------------------------
// Every kernel of a call is launched with programmatic stream serialization:
// it may be scheduled while its predecessor on the stream is still running.
// Each kernel therefore signals griddepcontrol.launch_dependents on entry and
// executes griddepcontrol.wait (which returns once the predecessor grid has
// completed and its memory is visible) before it reads anything an earlier
// launch wrote or writes anything at all.  Only reads of data no launch of a
// call writes (weights, tensor maps) may precede the wait.  KVR_PDL=0 in the
// environment turns the attribute off (every launch then waits in full).
bool pdl_enabled();

#ifdef __CUDACC__
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}
#endif
cudaError_t launch_prefix_match(const int32_t* slot_tokens, const int* slot_len, int n_slots,
                                int cap, const int32_t* prompt, int n, int32_t* out,
                                cudaStream_t st);
cudaError_t launch_gemv_int4(const GemvParams& p, int nt, cudaStream_t st);
cudaError_t launch_gemv_bf16(const GemvParams& p, int total_cols, cudaStream_t st);
cudaError_t launch_gemm_int4_tc(const GemmParams& p, int total_tiles, cudaStream_t st);
cudaError_t launch_attention(const AttnParams& p, int d, int row_warps, cudaStream_t st);
cudaError_t launch_attention_tc(const AttnParams& p, int d, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnParams& p, int d, cudaStream_t st);
// RoPE inverse frequencies theta^(-2j/d), j < d/2, in double (computed once
// per context on the host; d <= 128)
struct RopeFreq {
  double inv[64];
};
RopeFreq rope_freq(float theta, int d);
// table[i][j] = (cos, sin) of pos_i * inv[j], in double, rounded once to float
cudaError_t launch_rope_table(const RowMap& rows, int d, const RopeFreq& fr, float2* table,
                              cudaStream_t st);
// h = float(hidden) and the first RMSNorm: a = bf16(RMSNorm(h) * gain).
// Without a gain, a = hidden (attention-only layers; h untouched).  a16: a
// holds the bf16-rounded values as fp16 (the tcgen05 GEMM's operand type).
// The same launch writes the rows' RoPE table as launch_rope_table does.
// H must be a multiple of 8 (hidden, h and a rows 16-byte aligned).
cudaError_t launch_embed(const __nv_bfloat16* hidden, int m, int H, const __nv_bfloat16* gain,
                         float eps, float* h, __nv_bfloat16* a, bool a16, const RowMap& rows, int d,
                         const RopeFreq& fr, float2* table, cudaStream_t st);
// a = bf16(RMSNorm(h) * gain) for rows [0, m) of the fp32 residual stream
// (after a small-m residual projection, whose tiles each hold part of a row)
cudaError_t launch_norm(const float* h, int m, int H, const __nv_bfloat16* gain, float eps,
                        __nv_bfloat16* a, cudaStream_t st);
// out[t] = the row of the largest value over the tiles' bests of token t
// (lowest row on ties), t < m
// one device-side wait that runs out (the failure path, without a fault)
cudaError_t launch_wait_probe(int* status, cudaStream_t st);
// the persistent small-m pass (nt: tensor-core n-tiles of 8 rows, 1 or 2)
cudaError_t launch_pass(const PassParams& p, int nt, cudaStream_t st);
cudaError_t pass_setup();
int pass_ctas();   // CTAs of the pass (one per SM), 0 before pass_setup
cudaError_t launch_head_argmax(const float2* best, int tiles, int m, int32_t* out, cudaStream_t st);
cudaError_t launch_epi_qkv(const float* part, long long plane, int ksplit, int ldo, int c0,
                           int mb, const RowMap& rows, int Hq, int Hkv, int d,
                           const float2* rope, __nv_bfloat16* q, __nv_bfloat16* arena,
                           long long k_off, long long v_off, long long slot_stride, int cap,
                           cudaStream_t st);
// a16: a_out holds fp16 (as launch_embed); final_out is always bf16
cudaError_t launch_epi_resid(const float* part, long long plane, int ksplit, int ldo, int c0,
                             int mb, int H, float* h, const __nv_bfloat16* gain, float eps,
                             __nv_bfloat16* a_out, bool a16, __nv_bfloat16* final_out, cudaStream_t st);
cudaError_t launch_epi_swiglu(const float* part, long long plane, int ksplit, int ldo, int c0,
                              int mb, int F, __nv_bfloat16* z, cudaStream_t st);
// f16: out holds fp16 (a later layer's tcgen05 GEMM input)
cudaError_t launch_epi_cast(const float* part, long long plane, int ksplit, int ldo, int c0,
                            int mb, int N, __nv_bfloat16* out, bool f16, cudaStream_t st);

// dynamic shared memory the launchers need (for cudaFuncSetAttribute at setup)
// resident CTAs per SM of the int4 GEMV for nt token tiles, epilogue and weight format
int gemv_int4_per_sm(int nt, int epi, int fmt);
int attn_key_warps(int row_warps);   // consumer warps per row tile taking alternate key blocks
cudaError_t gemv_setup();
cudaError_t gemm_tc_setup();
cudaError_t attn_setup();
cudaError_t attn_tc_setup();
cudaError_t static_match_scratch(int32_t** prompt, int** slot_len, int32_t** match_out);

}  // namespace kvr

// ----------------------------------------------------------------------------
// device helpers (inline PTX)
// ----------------------------------------------------------------------------
#ifdef __CUDACC__
namespace kvr {
namespace dev {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Programmatic dependent launch: let the next kernel on the stream be
// scheduled, and wait for the previous one to complete.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test of a phase: try_wait may suspend the thread until the
// phase completes or a hardware time limit passes, so a thread that must go
// on with other work when the phase is not complete (and may itself be the
// one that completes it later) tests with test_wait instead.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The device status word: non-zero once any wait of any launch has given up.
__device__ __forceinline__ bool status_set(const int* status) {
  return status && *reinterpret_cast<const volatile int*>(status) != 0;
}

constexpr unsigned long long kStatusPollNs = 4000;
// Wait for the phase of `parity` to complete; give up after kWaitLimitNs,
// record the timeout in the device status word and return false.  A wait
// that finds the status word already set (another CTA, or an earlier launch,
// gave up) returns false at once, so one stall ends every CTA's waits
// within microseconds instead of one limit per wait.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  // the status word is read once every few microseconds of waiting: a global
  // load in the loop would otherwise delay noticing the phase
  unsigned long long next_check = t0 + kStatusPollNs;
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t = globaltimer_ns();
    if (t > next_check) {
      if (status_set(status)) return false;
      next_check = t + kStatusPollNs;
    }
    if (t - t0 > kWaitLimitNs) {
      if (status) atomicExch(status, kStatusTimeout);
      return false;
    }
  }
}

// Drain: wait for a phase until an absolute globaltimer deadline (one limit
// shared by all the stages a CTA drains before it exits).
__device__ __forceinline__ bool mbar_wait_until(uint32_t bar, uint32_t parity, unsigned long long deadline) {
  while (!mbar_try_wait(bar, parity))
    if (globaltimer_ns() > deadline) return false;
  return true;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled TMA load global -> shared, completion counted on an mbarrier.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* m, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Prefetch a 2-D tile into L2 (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* m, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(x), "r"(y)
               : "memory");
}

// Same with an L2 eviction-priority hint (weights are streamed once).
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* m, int x, int y,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                            uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                                  uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + C, fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float d[4], const uint32_t a[4], uint32_t b0,
                                               uint32_t b1, const float c[4]) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%10, %11, %12, %13};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
        "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// An activation pair rounded to bf16 (the model's rounding point), stored as
// bf16 or, for the tcgen05 GEMM's fp16 operands (f16), as the same two values
// in fp16: every bf16 number of magnitude 2^-14 .. 65504 is an fp16 number,
// so the conversion is exact there (smaller ones lose at most 2^-25).
__device__ __forceinline__ uint32_t pack_act2(float lo, float hi, bool f16) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  if (f16) {
    const float2 f = __bfloat1622float2(v);
    __half2 h = __floats2half2_rn(f.x, f.y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
  return *reinterpret_cast<uint32_t*>(&v);
}

// one activation, as pack_act2
__device__ __forceinline__ void store_act(__nv_bfloat16* dst, float x, bool f16) {
  const __nv_bfloat16 b = __float2bfloat16_rn(x);
  if (f16) *reinterpret_cast<__half*>(dst) = __float2half_rn(__bfloat162float(b));
  else *dst = b;
}

// *p += v at gpu scope with acquire-release semantics; returns the old value
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// 128-byte TMA swizzle: 16-byte chunk j of a 128-byte row r lands at j ^ (r % 8)
// (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace dev
}  // namespace kvr
#endif
