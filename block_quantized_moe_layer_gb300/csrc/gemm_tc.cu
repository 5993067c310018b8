// gemm_tc.cu -- grouped GEMM of the prefill-sized path on the tcgen05 tensor cores.
//
// One persistent CTA per SM (512 threads) claims work items from a global
// queue.  An item multiplies one 128-row tile of a block-quantized weight
// matrix (dequantised to bf16) by the bf16 activations of one token tile
// (n_pad <= 128 tokens), accumulating in fp32 in tensor memory:
//   warp 0      producer: 1-D bulk copies of the raw weight K-block and the
//               activation K-block into a 6-stage shared-memory ring;
//   warp 1      allocates the 512 TMEM columns; lane 0 issues the MMAs
//               (M = 128, N = n_pad, K = 16, A from TMEM, B from shared memory);
//   warps 4-11  dequantise: thread (row r, half h) turns its 32 weights of the
//               stage into bf16 pairs and stores them to TMEM (A operand);
//   warps 12-15 epilogue: read the accumulator (double-buffered in TMEM) and
//               write SwiGLU outputs (gate/up), bf16 partial outputs z (down) or
//               fp32 router logits.
// TMEM columns: A stages at 32 s (s < 6), accumulators at 256 and 384.
// Every wait is bounded; a timeout records its site in the status word, sets
// an abort flag that the other roles see, and every role then leaves after
// its own in-flight copies and MMAs have completed.
#include "large_t.cuh"
#include "tc.cuh"

namespace moe {

namespace {

constexpr int kStages = 6;
constexpr int kStageA = 16384;
constexpr int kStageBytes = 32768;
constexpr int kGemmThreads = 512;
constexpr int kDequantWarp0 = 4;
constexpr int kEpiWarp0 = 12;
constexpr int kTmemAcc = 256;

// dynamic shared-memory plan
constexpr int kOffStaging = kStages * kStageBytes;        // 4 warps x 4 KB
constexpr int kOffBars = kOffStaging + 4 * 4096;
constexpr int kNumBars = 3 * kStages + 2 + 2 + 4 + 4 + 1;
constexpr int kOffDescs = kOffBars + kNumBars * 8;
constexpr int kOffInfos = kOffDescs + kStages * 16;
constexpr int kOffMisc = kOffInfos + 4 * 48;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;          // + alignment slack

enum { kFlagEnd = 1, kFlagFirst = 2, kFlagLast = 4, kFlagHdr = 8 };

struct StageDesc {
  int flags, fmt, n_pad, kb;
};
struct ItemInfo {
  int end, kind, rt, e, slot0, n, n_pad, prow0, plane, pad[3];
};

enum { kSiteFree = 1, kSiteFull, kSiteDq, kSiteAcc, kSiteItem, kSiteDrain };

__device__ __forceinline__ void record_timeout(int* status, int site, int detail) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) {
    status[1] = site;
    status[2] = detail;
    status[3] = blockIdx.x;
  }
}

// Single-thread bounded wait.
__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t par, volatile int* abort, const LtGemmParams& p,
                                      int site, int detail) {
  uint64_t t0 = 0;
  while (!mbar_try_wait(bar, par)) {
    if (*abort) return false;
    const uint64_t now = globaltimer_ns();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > p.timeout_ns) {
      record_timeout(p.status, site, detail);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Whole-warp bounded wait with a warp-uniform result.
__device__ __forceinline__ bool waitw(uint64_t* bar, uint32_t par, volatile int* abort, const LtGemmParams& p,
                                      int site, int detail) {
  uint64_t t0 = 0;
  for (;;) {
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, par))) return true;
    int bail = 0;
    if ((threadIdx.x & 31) == 0) {
      if (*abort) {
        bail = 1;
      } else {
        const uint64_t now = globaltimer_ns();
        if (t0 == 0) {
          t0 = now;
        } else if (now - t0 > p.timeout_ns) {
          record_timeout(p.status, site, detail);
          *abort = 1;
          bail = 1;
        }
      }
    }
    if (__shfl_sync(0xffffffffu, bail, 0)) return false;
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 32 Q8_0 codes (8 words) times the block scale d -> 16 bf16 pairs.  A code
// byte b becomes the fp32 2^23 + (b ^ 0x80) by placing it under the exponent
// of 2^23; subtracting 2^23 + 128 recovers the signed code exactly, and
// q * d is exact in fp32 (8 x 11 significant bits); the only rounding is
// the conversion to bf16.
__device__ __forceinline__ void dq_q8(const uint4& a, const uint4& b, float d, uint32_t (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t f = w[i] ^ 0x80808080u;
    const float q0 = __int_as_float((int)__byte_perm(f, 0x4B000000u, 0x7440)) - 8388736.f;
    const float q1 = __int_as_float((int)__byte_perm(f, 0x4B000000u, 0x7441)) - 8388736.f;
    const float q2 = __int_as_float((int)__byte_perm(f, 0x4B000000u, 0x7442)) - 8388736.f;
    const float q3 = __int_as_float((int)__byte_perm(f, 0x4B000000u, 0x7443)) - 8388736.f;
    v[2 * i] = pack_bf16(q0 * d, q1 * d);
    v[2 * i + 1] = pack_bf16(q2 * d, q3 * d);
  }
}

// 32 Q4KS codes of one sub-block (16 bytes, weight 2j in the low nibble of
// byte j) -> 16 bf16 pairs of a*q - b, rounded once in fp32 (as the format
// defines it) and once to bf16.
__device__ __forceinline__ void dq_q4(const uint4& c, float a, float b, uint32_t (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float qe = __int_as_float((int)__byte_perm(lo, 0x4B000000u, 0x7440 + j)) - 8388608.f;
      const float qo = __int_as_float((int)__byte_perm(hi, 0x4B000000u, 0x7440 + j)) - 8388608.f;
      v[4 * i + j] = pack_bf16(fmaf(qe, a, -b), fmaf(qo, a, -b));
    }
  }
}

// 6-bit field f of a serialised Q4KS header (bits 32 + 6f .. of the 16 bytes).
__device__ __forceinline__ int q4_field(const uint32_t (&hw)[4], int f) {
  const int P = 32 + 6 * f, wi = P >> 5, sh = P & 31;
  uint32_t v = hw[wi] >> sh;
  if (sh > 26) v |= hw[wi + 1] << (32 - sh);
  return (int)(v & 63u);
}

__global__ void __launch_bounds__(kGemmThreads, 1) lt_gemm_kernel(const LtGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* full = bars;
  uint64_t* afull = bars + kStages;
  uint64_t* empty = bars + 2 * kStages;
  uint64_t* dfull = bars + 3 * kStages;
  uint64_t* dempty = dfull + 2;
  uint64_t* ifull = dempty + 2;
  uint64_t* iempty = ifull + 4;
  uint64_t* finbar = iempty + 4;
  StageDesc* descs = reinterpret_cast<StageDesc*>(sm + kOffDescs);
  ItemInfo* infos = reinterpret_cast<ItemInfo*>(sm + kOffInfos);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&afull[s], 8);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&dfull[a], 1);
      mbar_init(&dempty[a], 4);
    }
    for (int j = 0; j < 4; ++j) {
      mbar_init(&ifull[j], 1);
      mbar_init(&iempty[j], 4);
    }
    mbar_init(finbar, 1);
    *abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tc::alloc_512(tslot);
  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  const uint32_t tbase = *tslot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      uint32_t n = 0, i = 0;
      const int count = *p.n_items;
      int item = atomicAdd(p.queue, 1);
      bool ok = true;
      while (ok && item < count) {
        const int next = atomicAdd(p.queue, 1);
        const LtItem it = p.items[item];
        const LtTile tl = p.tiles[it.tile];
        const uint8_t* A;
        const uint8_t* B;
        int fmt, nkb;
        if (it.kind == kItemGU) {
          fmt = tl.e >= 0 ? p.fmt : p.sfmt;
          A = (tl.e >= 0 ? p.gu + (int64_t)tl.e * p.gu_stride : p.sgu) + it.rt * lt_tile_bytes(fmt, p.H);
          nkb = p.H / kLtKb;
          B = p.xg + (int64_t)tl.prow0 * p.H * 2;
        } else if (it.kind == kItemDN) {
          fmt = tl.e >= 0 ? p.fmt : p.sfmt;
          const int K = tl.e >= 0 ? p.I : p.Ish;
          A = (tl.e >= 0 ? p.dn + (int64_t)tl.e * p.dn_stride : p.sdn) + it.rt * lt_tile_bytes(fmt, K);
          nkb = K / kLtKb;
          B = p.h + (int64_t)tl.prow0 * p.Imax * 2;
        } else {
          fmt = MOE_BF16;
          A = p.router + it.plane * p.router_plane + it.rt * lt_tile_bytes(MOE_BF16, p.H);
          nkb = p.H / kLtKb;
          B = p.xg + (int64_t)tl.prow0 * p.H * 2;
        }
        // item information for the epilogue
        const uint32_t j = i & 3;
        if (i >= 4 && !(ok = wait1(&iempty[j], ((i >> 2) - 1) & 1, abort, p, kSiteItem, (int)i))) break;
        infos[j] = ItemInfo{0, it.kind, it.rt, tl.e, tl.slot0, tl.n, tl.n_pad, tl.prow0, it.plane, {0, 0, 0}};
        mbar_arrive(&ifull[j]);
        const uint32_t bbytes = (uint32_t)tl.n_pad * 128;
        for (int kb = 0; kb < nkb; ++kb, ++n) {
          const uint32_t s = n % kStages;
          if (n >= kStages && !(ok = wait1(&empty[s], ((n / kStages) - 1) & 1, abort, p, kSiteFree, (int)n))) break;
          uint8_t* sa = sm + s * kStageBytes;
          uint8_t* sb = sa + kStageA;
          int flags = (kb == 0 ? kFlagFirst : 0) | (kb == nkb - 1 ? kFlagLast : 0);
          const uint8_t* asrc;
          uint32_t abytes;
          if (fmt == MOE_Q8_0) {
            asrc = A + (int64_t)kb * kLtQ8Chunk;
            abytes = kLtQ8Chunk;
          } else if (fmt == MOE_Q4KS) {
            asrc = A + (int64_t)(kb >> 2) * kLtQ4Super + kLtQ4Hdr + (kb & 3) * kLtQ4Codes;
            abytes = kLtQ4Codes;
            if ((kb & 3) == 0) flags |= kFlagHdr;
          } else {
            asrc = A + (int64_t)kb * kLtBf16Chunk;
            abytes = kLtBf16Chunk;
          }
          descs[s] = StageDesc{flags, fmt, tl.n_pad, kb};
          const uint32_t hbytes = (flags & kFlagHdr) ? kLtQ4Hdr : 0;
          mbar_arrive_expect_tx(&full[s], abytes + hbytes + bbytes);
          bulk_g2s(sa, asrc, abytes, &full[s]);
          if (hbytes) bulk_g2s(sa + kLtQ4Codes, A + (int64_t)(kb >> 2) * kLtQ4Super, hbytes, &full[s]);
          bulk_g2s(sb, B + (int64_t)kb * bbytes, bbytes, &full[s]);
        }
        ++i;
        item = next;
      }
      // end markers
      if (ok) {
        const uint32_t j = i & 3;
        if (i < 4 || (ok = wait1(&iempty[j], ((i >> 2) - 1) & 1, abort, p, kSiteItem, (int)i))) {
          infos[j].end = 1;
          mbar_arrive(&ifull[j]);
        }
      }
      if (ok) {
        const uint32_t s = n % kStages;
        if (n < kStages || (ok = wait1(&empty[s], ((n / kStages) - 1) & 1, abort, p, kSiteFree, (int)n))) {
          descs[s].flags = kFlagEnd;
          mbar_arrive(&full[s]);
          ++n;
        }
      }
      // every copy this thread issued has landed before the CTA leaves
      const uint32_t n0 = n > kStages ? n - kStages : 0;
      for (uint32_t m = n0; m < n; ++m) {
        uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[m % kStages], (m / kStages) & 1)) {
          if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_timeout(p.status, kSiteDrain, (int)m);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      uint32_t n = 0, i = 0, a = 0;
      for (;; ++n) {
        const uint32_t s = n % kStages, par = (n / kStages) & 1;
        if (!wait1(&full[s], par, abort, p, kSiteFull, (int)n)) break;
        const StageDesc d = descs[s];
        if (d.flags & kFlagEnd) break;
        if (d.flags & kFlagFirst) {
          a = i & 1;
          const uint32_t u = i >> 1;
          if (u >= 1 && !wait1(&dempty[a], (u - 1) & 1, abort, p, kSiteAcc, (int)i)) break;
        }
        if (!wait1(&afull[s], par, abort, p, kSiteDq, (int)n)) break;
        tc::fence_after();
        const uint32_t idesc = tc::idesc_bf16(kLtRows, d.n_pad);
        const uint32_t bsm = smem_u32(sm + s * kStageBytes + kStageA);
        const uint32_t lbo = (uint32_t)d.n_pad * 16;
#pragma unroll
        for (int j = 0; j < kLtKb / 16; ++j) {
          const uint64_t bdesc = tc::smem_desc(bsm + j * 2 * lbo, lbo, 128);
          tc::mma_ts(tbase + kTmemAcc + 128 * a, tbase + 32 * s + 8 * j, bdesc, idesc,
                     ((d.flags & kFlagFirst) && j == 0) ? 0u : 1u);
        }
        tc::commit(&empty[s]);
        if (d.flags & kFlagLast) {
          tc::commit(&dfull[a]);
          ++i;
        }
      }
      // all MMAs of this thread complete before the accumulators are freed
      tc::commit(finbar);
      uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(finbar, 0)) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          record_timeout(p.status, kSiteDrain, -1);
          break;
        }
      }
    }
  } else if (warp >= kDequantWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------------ dequantise
    const int q = warp & 3, h = (warp - kDequantWarp0) >> 2, r = 32 * q + lane;
    uint32_t hw[4] = {0, 0, 0, 0};
    for (uint32_t n = 0;; ++n) {
      const uint32_t s = n % kStages, par = (n / kStages) & 1;
      if (!waitw(&full[s], par, abort, p, kSiteFull, (int)n)) break;
      const StageDesc d = descs[s];
      if (d.flags & kFlagEnd) break;
      // the MMAs that read this TMEM stage last time have completed
      if (n >= kStages && !waitw(&empty[s], ((n / kStages) - 1) & 1, abort, p, kSiteFree, (int)n)) break;
      tc::fence_after();
      const uint8_t* sa = sm + s * kStageBytes;
      uint32_t v[16];
      if (d.fmt == MOE_Q8_0) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(sa + ((h * 2 + 0) * 128 + r) * 16);
        const uint4 c1 = *reinterpret_cast<const uint4*>(sa + ((h * 2 + 1) * 128 + r) * 16);
        const float dsc = __half2float(*reinterpret_cast<const __half*>(sa + 8192 + (h * 128 + r) * 2));
        dq_q8(c0, c1, dsc, v);
      } else if (d.fmt == MOE_Q4KS) {
        if (d.flags & kFlagHdr) {
          const uint4 hv = *reinterpret_cast<const uint4*>(sa + kLtQ4Codes + r * 16);
          hw[0] = hv.x; hw[1] = hv.y; hw[2] = hv.z; hw[3] = hv.w;
        }
        const int sub = 2 * (d.kb & 3) + h;
        const float dd = __half2float(__ushort_as_half((unsigned short)(hw[0] & 0xFFFFu)));
        const float dm = __half2float(__ushort_as_half((unsigned short)(hw[0] >> 16)));
        const float av = dd * (float)q4_field(hw, sub);
        const float bv = dm * (float)q4_field(hw, 8 + sub);
        const uint4 c = *reinterpret_cast<const uint4*>(sa + (h * 128 + r) * 16);
        dq_q4(c, av, bv, v);
      } else {
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
          const uint4 c = *reinterpret_cast<const uint4*>(sa + ((h * 4 + pc) * 128 + r) * 16);
          v[4 * pc + 0] = c.x; v[4 * pc + 1] = c.y; v[4 * pc + 2] = c.z; v[4 * pc + 3] = c.w;
        }
      }
      tc::st_32x32b_x16(tbase + ((uint32_t)(32 * q) << 16) + 32 * s + 16 * h, v);
      tc::wait_st();
      tc::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&afull[s]);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3, r = 32 * q + lane;
    uint8_t* stg = sm + kOffStaging + q * 4096;
    for (uint32_t i = 0;; ++i) {
      const uint32_t j = i & 3;
      if (!waitw(&ifull[j], (i >> 2) & 1, abort, p, kSiteItem, (int)i)) break;
      const ItemInfo info = infos[j];
      if (info.end) break;
      const uint32_t a = i & 1;
      if (!waitw(&dfull[a], (i >> 1) & 1, abort, p, kSiteAcc, (int)i)) break;
      tc::fence_after();
      const uint32_t tacc = tbase + ((uint32_t)(32 * q) << 16) + kTmemAcc + 128 * a;
      for (int c = 0; c < info.n_pad; c += 16) {
        uint32_t v[16];
        tc::ld_32x32b_x16(tacc + c, v);
        tc::wait_ld();
        if (info.kind == kItemGU) {
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float g = __uint_as_float(v[m]);
            const float u = __shfl_down_sync(0xffffffffu, g, 16);
            if (lane < 16) {
              const float hv = g / (1.f + expf(-g)) * u;
              const int nn = c + m;
              *reinterpret_cast<__nv_bfloat16*>(stg + ((lane >> 3) * info.n_pad + nn) * 16 + (lane & 7) * 2) =
                  __float2bfloat16_rn(hv);
            }
          }
        } else if (info.kind == kItemDN) {
          const int o = kLtRows * info.rt + r;
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            if (c + m < info.n)
              p.z[(int64_t)(info.slot0 + c + m) * p.H + o] = __float2bfloat16_rn(__uint_as_float(v[m]));
          }
        } else {
          const int e = kLtRows * info.rt + r;
          const int t0 = info.slot0 - p.T * p.k;
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            if (c + m < info.n)
              p.logits[((int64_t)info.plane * p.T + t0 + c + m) * p.E_pad128 + e] = __uint_as_float(v[m]);
          }
        }
      }
      tc::fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&dempty[a]);
        mbar_arrive(&iempty[j]);
      }
      if (info.kind == kItemGU) {
        // this warp's two column chunks of the h K-block are one contiguous range
        const int nv = 2 * info.n_pad;  // 16-byte vectors
        uint4* dst = reinterpret_cast<uint4*>(p.h + (int64_t)info.prow0 * p.Imax * 2 +
                                              (int64_t)info.rt * info.n_pad * 128 + (int64_t)2 * q * info.n_pad * 16);
        const uint4* src = reinterpret_cast<const uint4*>(stg);
        for (int x = lane; x < nv; x += 32) dst[x] = src[x];
        __syncwarp();
      }
    }
  }

  tc::fence_before();
  __syncthreads();
  tc::fence_after();
  if (warp == 1) tc::dealloc_512(tbase);
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(p.exit_cnt, 1) == (int)gridDim.x - 1) {
      *p.queue = 0;
      *p.exit_cnt = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t lt_gemm_configure() {
  return cudaFuncSetAttribute(lt_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t lt_gemm_launch(const LtGemmParams& p, int grid, cudaStream_t st) {
  lt_gemm_kernel<<<grid, kGemmThreads, kSmemBytes, st>>>(p);
  return cudaGetLastError();
}

}  // namespace moe
