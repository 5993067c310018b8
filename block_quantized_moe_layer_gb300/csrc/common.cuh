// common.cuh -- device helpers and the internal weight / activation layouts.
#pragma once
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <algorithm>

#include "../../include/moe_layer.h"

namespace moe {

// ---------------------------------------------------------------------------
// Tiling constants of the small-T (GEMV) path.
//   A weight chunk holds 32 rows (one per lane) x Kc columns of one matrix; the
//   8 consumer warps split the chunk's 32-column blocks between them.
// ---------------------------------------------------------------------------
constexpr int kRows = 32;           // rows per chunk (= lanes)
constexpr int kConsumerWarps = 8;   // warps that compute (warps 0-7)
constexpr int kProducerWarp = 8;    // issues the bulk copies (one thread)
constexpr int kEpilogueWarp = 9;    // reduces finished row groups, does the bookkeeping
constexpr int kThreads = 10 * 32;
constexpr int kGroup = 4;           // activation vectors per tile (token group)
constexpr int kBlocksPerStep = kConsumerWarps;        // consumer warp w takes blocks w, w + 8, ...
constexpr int kRouterKc = 256;      // router repack block columns
constexpr int kRouterCc = 128;      // router chunk columns (half a repack block)
constexpr int kRouterTileChunks = 4;  // router chunks per router tile (512 columns)
constexpr int kQ8KcMax = 2048;      // largest Q8_0 chunk (columns)
constexpr int kQ4KcMax = 4096;      // largest Q4KS chunk (columns)
constexpr int kMaxSmallT = 8;       // largest T of the GEMV path
constexpr int kMaxTopK = 16;        // largest top_k
constexpr int kMaxE = 1024;         // largest expert count
constexpr int kMaxDownTiles = 256;  // largest H / 128
constexpr int kMaxSlots = 8;        // stage descriptor slots of the small-T ring

// Activation record of one 32-value block: L limb planes of 32 bytes each
// (byte i of limb l = bits [8l, 8l+8) of the block fixed-point integer X_i,
// lower limbs unsigned, the top limb signed), then fp32 ascale = 2^-s and
// fp32 sumx = ascale * sum_i X_i, then 8 bytes of padding.  X_i =
// round(v_i * 2^s) with s chosen so that max |X_i| <= 2^(8L-2).
__host__ __device__ constexpr int rec_bytes(int L) { return 32 * L + 16; }

// Bytes of one weight chunk: 32 rows x Kc columns (nbc = Kc/32 blocks).
//   Q8_0 : quants [nbc][2 halves][32 rows][16 B], then scales [nbc][32 rows] fp16
//   Q4KS : quants [nbc sub-blocks][32 rows][16 B] (nibbles permuted so that
//          (word & 0x0F0F0F0F) holds weights 8w..8w+3 and
//          ((word >> 4) & 0x0F0F0F0F) weights 8w+4..8w+7), then the
//          serialised 16-byte superblock headers [nbc/8][32 rows][16 B]
//   F32  : [Kc/4][32 rows][4 floats]   (router; lane = row)
__host__ __device__ inline int64_t chunk_bytes(int fmt, int Kc) {
  if (fmt == MOE_Q8_0) return (int64_t)(Kc / 32) * 1088;
  if (fmt == MOE_Q4KS) return (int64_t)(Kc / 32) * 512 + (int64_t)(Kc / 256) * 512;
  return (int64_t)Kc * kRows * 4;
}

// Chunking of a reduction dimension K for a format: n chunks of Kc columns,
// Kc at most the format's largest chunk >> shift (shift > 0 when shared
// memory cannot hold two stages of the largest chunks).
struct Chunking {
  int n, Kc;
};
inline Chunking choose_chunking(int fmt, int K, int shift = 0) {
  const int unit = fmt == MOE_Q4KS ? 256 : (fmt == MOE_Q8_0 ? 32 : kRouterKc);
  const int kmax = std::max(unit, (fmt == MOE_Q4KS ? kQ4KcMax : (fmt == MOE_Q8_0 ? kQ8KcMax : kRouterKc)) >> shift);
  int n = (K + kmax - 1) / kmax;
  for (; n <= K / unit; ++n)
    if (K % n == 0 && (K / n) % unit == 0) return {n, K / n};
  return {0, 0};
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Waits for the phase with the given parity; the thread may be suspended (it
// takes no issue slots) for up to 0.5 ms before the call returns false.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(500000)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes and
// both addresses must be multiples of 16).
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// An L2 policy that marks lines as first to evict: for data read once per
// launch (streamed weights), so that it does not push out the small working
// set (counters, records, outputs) that the CTAs exchange through L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Programmatic dependent launch: let the next kernel in the stream (launched
// with programmatic stream serialization) start its CTAs early, and wait for
// the previous kernel's completion and memory before reading what it wrote.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launches a kernel with programmatic stream serialization (it must call
// griddep_wait before reading anything an earlier kernel in the stream wrote).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}


// bulk_g2s with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void* dst_smem, const void* src, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Phase stamp: word w keeps the maximum of t ("last" events) or of ~t
// ("first" events).
__device__ __forceinline__ void stamp_last(unsigned long long* st, int w) {
  atomicMax(st + w, (unsigned long long)globaltimer_ns());
}
__device__ __forceinline__ void stamp_first(unsigned long long* st, int w) {
  atomicMax(st + w, ~(unsigned long long)globaltimer_ns());
}
__device__ __forceinline__ void stamp_first_at(unsigned long long* st, int w, uint64_t t) {
  atomicMax(st + w, ~(unsigned long long)t);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// A strong (relaxed, GPU scope) 64-bit load: every call reads the word anew.
__device__ __forceinline__ long long ld_relaxed_s64(const long long* p) {
  long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Add with release semantics at GPU scope (no value returned).
__device__ __forceinline__ void red_add_release(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Fetch-and-add with acquire and release semantics at GPU scope.
__device__ __forceinline__ int atom_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Orders this thread's generic-proxy global accesses with its async-proxy
// (bulk copy) accesses: records written with st.global by one CTA and read
// with cp.async.bulk by another need it on both sides of the flag hand-off.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Named barrier over the consumer warps only (the producer warp keeps going).
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// The same barrier, returning whether any consumer thread passed true.
__device__ __forceinline__ bool consumer_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, %2, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}

// dp4a variants: a = weight bytes, b = activation limb bytes.
__device__ __forceinline__ int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Scale of the block sum in a record: sum(X) * 2^-s in fp32, rounded once.
// The integer sum is exact; for L = 2 it fits fp32's mantissa (|sum| < 2^20),
// and the scaling by a power of two is exact (no subnormal results: s <= 120).
__device__ __forceinline__ float record_sumx(long long sx, int s) { return ldexpf(__ll2float_rn(sx), -s); }

// One warp converts 32 values (lane i holds v) into an activation record.
template <int L>
__device__ __forceinline__ void write_record(float v, uint8_t* rec) {
  const int lane = threadIdx.x & 31;
  const float amax = warp_max(fabsf(v));
  int s = 0;
  if (amax > 0.f) {
    s = (8 * L - 3) - ilogbf(amax);
    s = max(-100, min(120, s));
  }
  const int X = __float2int_rn(ldexpf(v, s));
#pragma unroll
  for (int l = 0; l < L; ++l) rec[l * 32 + lane] = (uint8_t)((X >> (8 * l)) & 0xFF);
  long long sx;
  if constexpr (L == 2) {
    sx = __reduce_add_sync(0xffffffffu, X);  // |X| <= 2^14: the sum fits 32 bits
  } else {
    sx = X;
#pragma unroll
    for (int o = 16; o; o >>= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
  }
  if (lane == 0)
    *reinterpret_cast<float4*>(rec + 32 * L) = make_float4(ldexpf(1.f, -s), record_sumx(sx, s), 0.f, 0.f);
}

// The same record as write_record, written by one thread from the block's 32
// values v (rec 16-byte aligned).  The arithmetic is the same, so the bytes
// are the same.
template <int L>
__device__ __forceinline__ void record_from_values(const float (&v)[32], uint8_t* rec) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  int s = 0;
  if (amax > 0.f) {
    s = (8 * L - 3) - ilogbf(amax);
    s = max(-100, min(120, s));
  }
  long long sx = 0;
  uint32_t packed[L][8];
#pragma unroll
  for (int l = 0; l < L; ++l)
#pragma unroll
    for (int j = 0; j < 8; ++j) packed[l][j] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int X = __float2int_rn(ldexpf(v[i], s));
    sx += X;
#pragma unroll
    for (int l = 0; l < L; ++l) packed[l][i >> 2] |= (uint32_t)((X >> (8 * l)) & 0xFF) << (8 * (i & 3));
  }
#pragma unroll
  for (int l = 0; l < L; ++l) {
    uint4* d = reinterpret_cast<uint4*>(rec + 32 * l);
    d[0] = make_uint4(packed[l][0], packed[l][1], packed[l][2], packed[l][3]);
    d[1] = make_uint4(packed[l][4], packed[l][5], packed[l][6], packed[l][7]);
  }
  *reinterpret_cast<float4*>(rec + 32 * L) =
      make_float4(ldexpf(1.f, -s), record_sumx(sx, s), 0.f, 0.f);
}

// The record of one block of 32 values read from shared memory (bf16 for
// L = 2, fp32 for L = 4), by one thread.
template <int L>
__device__ __forceinline__ void write_record_lane(const uint8_t* src, uint8_t* rec) {
  float v[32];
#pragma unroll
  for (int q = 0; q < (L == 2 ? 4 : 8); ++q) {
    const uint4 u = reinterpret_cast<const uint4*>(src)[q];
    if constexpr (L == 2) {
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        v[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
        v[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    } else {
      v[4 * q] = __uint_as_float(u.x);
      v[4 * q + 1] = __uint_as_float(u.y);
      v[4 * q + 2] = __uint_as_float(u.z);
      v[4 * q + 3] = __uint_as_float(u.w);
    }
  }
  record_from_values<L>(v, rec);
}

// Status bits written into the layer's status word.
constexpr int kStatusTimeout = 1;

}  // namespace moe
