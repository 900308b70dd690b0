// Prefix match on the device: longest common token prefix of every occupied
// slot with the prompt, and of every pair of occupied slots.
//
// goinfer, "Turn nine in under half a second" ("How it works"): the prompt
// goes to the slot with the longest common token prefix, provided that prefix
// exceeds the longest one the slot has in common with any other slot.  Both
// quantities are
// first-mismatch positions; one CTA computes one of them by scanning its two
// token rows in 256-token chunks and stopping at the first chunk that holds a
// mismatch (block-wide vote, then a shared-memory minimum).
#include <climits>

#include "kvr_internal.cuh"

namespace kvr {

namespace {

__global__ void prefix_match_kernel(const int32_t* slot_tokens, const int* slot_len, int n_slots,
                                    int cap, const int32_t* prompt, int n, int32_t* out) {
  const int a = blockIdx.y;  // slot
  const int b = blockIdx.x;  // other slot, or n_slots for the prompt
  if (b != n_slots && b <= a) return;
  __shared__ int first;
  const int la = slot_len[a];
  const int lb = b == n_slots ? n : slot_len[b];
  int L = (la < 0 || lb < 0) ? 0 : min(la, lb);
  const int32_t* A = slot_tokens + (long long)a * cap;
  const int32_t* B = b == n_slots ? prompt : slot_tokens + (long long)b * cap;
  if (threadIdx.x == 0) first = L;
  __syncthreads();
  for (int base = 0; base < L; base += blockDim.x) {
    const int idx = base + threadIdx.x;
    const bool mm = idx < L && A[idx] != B[idx];
    if (__syncthreads_or(mm)) {
      if (mm) atomicMin(&first, idx);
      __syncthreads();
      break;
    }
  }
  if (threadIdx.x == 0) out[a * (n_slots + 1) + b] = first;
}

}  // namespace

cudaError_t launch_prefix_match(const int32_t* slot_tokens, const int* slot_len, int n_slots,
                                int cap, const int32_t* prompt, int n, int32_t* out,
                                cudaStream_t st) {
  const dim3 grid(n_slots + 1, n_slots);
  prefix_match_kernel<<<grid, 256, 0, st>>>(slot_tokens, slot_len, n_slots, cap, prompt, n, out);
  return cudaGetLastError();
}

}  // namespace kvr
