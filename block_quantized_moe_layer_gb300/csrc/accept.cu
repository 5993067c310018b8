// accept.cu -- greedy draft acceptance over the verify batch.
//
// "Support Step3.5/3.7 flash mtp3" (llama.cpp PR #24340), "Overview", Round 1
// steps 4-5: the target's token for verify row i is compared with draft
// i+1; the first mismatch stops acceptance and the target's token there is
// the next token.  Greedy sampling = argmax, ties to the lowest token id.
//
// Each of the (k+1) rows is split over S CTAs; each CTA writes its partial
// (max, argmax) to the caller's workspace, and the last CTA to finish (a
// counter in the workspace) reduces the partials in split order, counts the
// matching prefix and writes the two outputs.  The counter is left at zero.
//
// Inside an MTP round the last CTA also applies the draft confidence cut
// ("Step-3.5-Flash MTP GGUF", "Usage": --spec-draft-p-min): given each
// draft's probability under its own logits, drafting stopped at the first
// draft below p_min, so that draft and every later one become -1 (they match
// no token, which ends the accepted prefix there).

#include "common.cuh"

namespace moe {

constexpr int kAcceptThreads = 256;
constexpr int kAcceptSplitCols = 16384;

int accept_splits(int V) {
  int s = (V + kAcceptSplitCols - 1) / kAcceptSplitCols;
  return s < 1 ? 1 : (s > 64 ? 64 : s);
}

struct ArgPart {
  float v;
  int i;
};

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(const int32_t* __restrict__ draft, int k,
                                                                const float* __restrict__ logits, int V, int S,
                                                                int32_t* out_n, int32_t* out_next,
                                                                int* counter, ArgPart* parts,
                                                                const float* __restrict__ dprob, float p_min,
                                                                int32_t* draft_cut) {
  __shared__ float sv[kAcceptThreads / 32];
  __shared__ int si[kAcceptThreads / 32];
  __shared__ int last;
  griddep_launch_dependents();
  griddep_wait();  // the logits and drafts may come from the previous kernel in the stream
  const int row = blockIdx.x / S, sp = blockIdx.x % S;
  const int per = (V + S - 1) / S;
  const int c0 = sp * per, c1 = min(V, c0 + per);
  const float* lr = logits + (int64_t)row * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  for (int c = c0 + threadIdx.x; c < c1; c += kAcceptThreads) {
    const float v = __ldg(lr + c);
    if (v > bv) { bv = v; bi = c; }  // increasing c: strict > keeps the lowest index
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kAcceptThreads / 32; ++w)
      if (better(sv[w], si[w], bv, bi)) { bv = sv[w]; bi = si[w]; }
    parts[blockIdx.x] = ArgPart{bv, bi};
    __threadfence();
    last = (atomicAdd(counter, 1) == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (!last || threadIdx.x != 0) return;
  __threadfence();
  int kk = k;  // drafts kept by the confidence cut
  if (dprob) {
    for (int j = 0; j < k; ++j)
      if (!(dprob[j] >= p_min)) {
        kk = j;
        break;
      }
    for (int j = kk; j < k; ++j) draft_cut[j] = -1;
  }
  int n = 0;
  bool run = true;
  int a_n = 0;
  for (int r = 0; r <= kk; ++r) {
    float rv = -INFINITY;
    int ri = 0x7fffffff;
    for (int s = 0; s < S; ++s) {
      const float v = __ldcg(&parts[r * S + s].v);
      const int i = __ldcg(&parts[r * S + s].i);
      if (better(v, i, rv, ri)) { rv = v; ri = i; }
    }
    if (run) {
      if (r < kk && ri == draft[r]) {
        ++n;
      } else {
        a_n = ri;
        run = false;
      }
    }
  }
  *out_n = n;
  *out_next = a_n;
  *counter = 0;
  __threadfence();
}

size_t accept_workspace_bytes(int k, int V) { return 16 + (size_t)(k + 1) * accept_splits(V) * sizeof(ArgPart); }

cudaError_t accept_launch(const int32_t* draft, int k, const float* logits, int V, int32_t* out_n,
                          int32_t* out_next, void* ws, cudaStream_t st) {
  const int S = accept_splits(V);
  int* counter = static_cast<int*>(ws);
  ArgPart* parts = reinterpret_cast<ArgPart*>(static_cast<uint8_t*>(ws) + 16);
  return launch_pdl(accept_kernel, (k + 1) * S, kAcceptThreads, 0, st, draft, k, logits, V, S, out_n, out_next,
                    counter, parts, (const float*)nullptr, 0.f, (int32_t*)nullptr);
}

// The same with the draft confidence cut: dprob[k] the drafts' probabilities;
// drafts from the first one below p_min on are set to -1 in `draft`.
cudaError_t accept_launch_cut(int32_t* draft, int k, const float* logits, int V, const float* dprob, float p_min,
                              int32_t* out_n, int32_t* out_next, void* ws, cudaStream_t st) {
  const int S = accept_splits(V);
  int* counter = static_cast<int*>(ws);
  ArgPart* parts = reinterpret_cast<ArgPart*>(static_cast<uint8_t*>(ws) + 16);
  return launch_pdl(accept_kernel, (k + 1) * S, kAcceptThreads, 0, st, (const int32_t*)draft, k, logits, V, S, out_n,
                    out_next, counter, parts, dprob, p_min, draft);
}

// Scratch of the allocation-free entry point (mtp_verify_accept_noalloc).
// A C runtime that drives the draft/verify loop itself may hold no device
// allocator at all (no torch, no pool), and cudaMalloc / cudaFree would
// synchronise the device between two verify rounds, so that caller gets a
// fixed scratch that lives in the library's own module instead.  Every call
// on a device uses this one array: the counter at its start must be zero
// when a call begins (it is zero at module load and every completed call
// leaves it at zero); the partials behind it are written before they are
// read.  Two calls whose kernels overlap on the GPU race on it.
constexpr size_t kAcceptStaticBytes = 4096;
static __device__ __align__(256) uint8_t g_accept_scratch[kAcceptStaticBytes];

size_t accept_static_bytes() { return kAcceptStaticBytes; }

// Device address of g_accept_scratch in the current device's context.  The
// host-side name of the array is only a stand-in, so the address is asked of
// the runtime with that device current.  It is looked up on every call
// rather than cached: a cached address would outlive the context it belongs
// to (cudaDeviceReset tears the context down and the module is loaded again,
// possibly elsewhere, in the next one), while the lookup itself is a host-side
// table read once the module is loaded.  The first lookup on a device loads
// the library's module there, so the first call on a device belongs before
// any stream capture on it.
cudaError_t accept_static_scratch(void** out) {
  void* p = nullptr;
  const cudaError_t rc = cudaGetSymbolAddress(&p, g_accept_scratch);
  if (rc != cudaSuccess) return rc;
  *out = p;
  return cudaSuccess;
}

}  // namespace moe
