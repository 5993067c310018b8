// gemm_tc.cu -- grouped GEMM of the prefill-sized path on the tcgen05 tensor cores.
//
// One persistent CTA per SM (512 threads) claims work items from a global
// queue.  An item multiplies one 128-row tile of a block-quantized weight
// matrix (dequantised to fp16) by the fp16 activations of one token tile
// (n_pad <= 64 tokens), accumulating in fp32 in tensor memory (TMEM).
//   warp 0      producer: 1-D bulk copies of raw weight stages (A ring) and
//               activation K-slices (B ring);
//   warp 1      allocates the 512 TMEM columns; lane 0 issues the MMAs
//               (M = 128, N = n_pad, K = 16, A from TMEM, B from shared memory);
//   warps 4-11  dequantise, as two groups of four warps that share every A
//               stage: thread (group g, row r) turns its row's weights in
//               half g of the stage into fp16 pairs and stores them to TMEM;
//   warps 12-15 epilogue: read the accumulator (double-buffered) and write
//               SwiGLU outputs (gate/up), bf16 partial outputs z (down) or fp32
//               router logits.
// The three rings are released independently: a raw weight slot as soon as
// both groups hold its data in registers, an activation slot and a TMEM stage
// when the MMAs that read them complete.  An A stage is 256 columns of Q8_0,
// one 256-column superblock of Q4KS or 128 columns of a router plane, and
// fills one TMEM stage of 128 columns (up to 16 MMAs).
// TMEM columns: A stages at 128 s (s < 2), accumulators at 384 and 448.
// Every wait is bounded; a timeout records its site in the status word, sets
// an abort flag that the other roles see, and every role then leaves after
// its own in-flight copies and MMAs have completed.
#include "large_t.cuh"
#include "tc.cuh"

namespace moe {

namespace {

// A stage covers up to 256 columns of K: one TMEM stage of 128 columns (16
// MMAs of K = 16), so the issuer's fixed cost per stage (its waits, one
// commit, its bookkeeping: ~700 cycles on a thread that shares its
// scheduler with busy warps) is spread over 16 MMAs.
constexpr int kStageK = 256;
constexpr int kTmemStage = kStageK / 2;  // TMEM columns of one A stage (two fp16 per column)
// Both dequant groups work on every stage (each on half of its blocks), so
// every waiter sees every phase of every ring in order, whatever the ring
// sizes.
constexpr int kNA = 3;            // raw weight slots
constexpr int kNT = 3;            // TMEM A stages
// activation slots: one per TMEM stage, indexed alike, so one MMA commit per
// stage frees both (a commit costs the tensor pipe ~80 cycles, about two
// small MMAs)
constexpr int kNB = kNT;
constexpr int kASlot = 4 * kLtQ8Chunk;  // 34816: Q8_0 (256 columns) >= two router K-blocks >= a Q4KS superblock
constexpr int kBSlot = kLtMaxN * kStageK * 2;
static_assert(kNT * kTmemStage <= 384, "A stages below the accumulators");
constexpr int kGemmThreads = 512;
constexpr int kDequantWarp0 = 4;
constexpr int kEpiWarp0 = 12;
constexpr int kTmemAcc = 384;

// dynamic shared-memory plan
constexpr int kOffB = kNA * kASlot;
constexpr int kOffStaging = kOffB + kNB * kBSlot;          // 4 warps x 2 chunks x 64 rows x 16 B
constexpr int kOffBars = kOffStaging + 4 * 2048;
constexpr int kNumBars = 2 * kNA + kNB + 2 * kNT + 2 + 2 + 4 + 4 + 1;
constexpr int kOffDescs = kOffBars + kNumBars * 8;
constexpr int kOffTdescs = kOffDescs + kNA * 48;
constexpr int kOffInfos = kOffTdescs + kNT * 16;
constexpr int kOffMisc = kOffInfos + 4 * 48;
constexpr int kSmemBytes = kOffMisc + 16 + 1024;          // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory plan");

enum { kFlagEnd = 1, kFlagFwdEnd = 2, kFlagFirst = 4, kFlagLast = 8 };

struct StageDesc {  // one A stage
  int flags, fmt, n_pad, cols, nt0, nts, tflags[2], pad[4];
};
struct TDesc {  // one TMEM stage, for the MMA issuer
  int flags, n_pad, nk, pad;
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

// Waits spin on the non-blocking test first (a suspended thread takes a few
// hundred cycles to resume, which would sit on the per-stage critical path),
// then fall back to the suspending try_wait.
constexpr int kSpin = 32;

// Single-thread bounded wait.
__device__ __forceinline__ bool wait1(uint64_t* bar, uint32_t par, volatile int* abort, const LtGemmParams& p,
                                      int site, int detail) {
  for (int i = 0; i < kSpin; ++i)
    if (mbar_test_wait(bar, par)) return true;
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
                                      int site, int detail, int spin = kSpin) {
  for (int i = 0; i < spin; ++i)
    if (__all_sync(0xffffffffu, mbar_test_wait(bar, par))) return true;
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

__device__ __forceinline__ uint64_t pack2(float a) {
  const uint32_t u = __float_as_uint(a);
  return ((uint64_t)u << 32) | u;
}

// Two Q4KS codes as 2^23 + q: w = a*q - b with one fp32 rounding (as the
// format defines it), then fp16.
__device__ __forceinline__ uint32_t q4_pair(uint32_t m0, uint32_t m1, uint64_t c2, uint64_t a2, uint64_t nb2) {
  uint32_t out;
  asm("{\n\t.reg .b64 x;\n\t.reg .b32 lo, hi;\n\t"
      "mov.b64 x, {%1, %2};\n\t"
      "sub.rn.f32x2 x, x, %3;\n\t"
      "fma.rn.f32x2 x, x, %4, %5;\n\t"
      "mov.b64 {lo, hi}, x;\n\t"
      "cvt.rn.f16x2.f32 %0, hi, lo;\n\t}"
      : "=r"(out)
      : "r"(m0), "r"(m1), "l"(c2), "l"(a2), "l"(nb2));
  return out;
}

// 32 Q8_0 codes (8 words; the LT copy holds each code byte with its sign bit
// flipped, u = q + 128) of one block with fp16 scale d -> 16 fp16 pairs.
// A byte permute places u under the fp16 exponent of 1024 (0x64uu = 1024 + u),
// subtracting 1152 gives q exactly, and the multiply by d rounds once:
// fp16(q * d).
__device__ __forceinline__ void dq_q8(const uint4& a, const uint4& b, uint32_t d2, uint32_t (&v)[16]) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  const __half2 c = __half2half2(__ushort_as_half((unsigned short)0x6480u));  // 1152
  const __half2 dd = *reinterpret_cast<const __half2*>(&d2);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    uint32_t lo = __byte_perm(w[i], 0x64646464u, 0x5140), hi = __byte_perm(w[i], 0x64646464u, 0x7362);
    const __half2 ql = __hsub2(*reinterpret_cast<const __half2*>(&lo), c);
    const __half2 qh = __hsub2(*reinterpret_cast<const __half2*>(&hi), c);
    const __half2 xl = __hmul2(ql, dd), xh = __hmul2(qh, dd);
    v[2 * i] = *reinterpret_cast<const uint32_t*>(&xl);
    v[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&xh);
  }
}

// 32 Q4KS codes of one sub-block (16 bytes, weight 2j in the low nibble of
// byte j) -> 16 fp16 pairs of a*q - b.
__device__ __forceinline__ void dq_q4(const uint4& c, float a, float b, uint32_t (&v)[16]) {
  const uint32_t w[4] = {c.x, c.y, c.z, c.w};
  const uint64_t c2 = pack2(8388608.f), a2 = pack2(a), nb2 = pack2(-b);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      v[4 * i + j] = q4_pair(__byte_perm(lo, 0x4B000000u, 0x7440 + j), __byte_perm(hi, 0x4B000000u, 0x7440 + j),
                             c2, a2, nb2);
  }
}

// 6-bit field f of a serialised Q4KS header (bits 32 + 6f .. of the 16 bytes;
// w1..w3 are its words 1..3).
__device__ __forceinline__ int q4_field(uint32_t w1, uint32_t w2, uint32_t w3, int f) {
  const int P = 6 * f;
  if (P < 32) {
    const uint64_t lo = ((uint64_t)w2 << 32) | w1;
    return (int)((lo >> P) & 63u);
  }
  const uint64_t hi = ((uint64_t)w3 << 32) | w2;
  return (int)((hi >> (P - 32)) & 63u);
}

__global__ void __launch_bounds__(kGemmThreads, 1) lt_gemm_kernel(const LtGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffBars);
  uint64_t* afull = bars;
  uint64_t* aempty = afull + kNA;
  uint64_t* bfull = aempty + kNA;
  uint64_t* tfull = bfull + kNB;
  uint64_t* tempty = tfull + kNT;
  uint64_t* dfull = tempty + kNT;
  uint64_t* dempty = dfull + 2;
  uint64_t* ifull = dempty + 2;
  uint64_t* iempty = ifull + 4;
  uint64_t* finbar = iempty + 4;
  StageDesc* descs = reinterpret_cast<StageDesc*>(sm + kOffDescs);
  TDesc* tdescs = reinterpret_cast<TDesc*>(sm + kOffTdescs);
  ItemInfo* infos = reinterpret_cast<ItemInfo*>(sm + kOffInfos);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
  volatile int* abort = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kNA; ++s) {
      mbar_init(&afull[s], 1);
      mbar_init(&aempty[s], 8);  // both dequant groups
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&bfull[s], 1);
    }
    for (int s = 0; s < kNT; ++s) {
      mbar_init(&tfull[s], 8);  // both dequant groups
      mbar_init(&tempty[s], 1);
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
  // setup only above: the previous kernel in the stream wrote the items,
  // operands and counters read below (or reads what this one writes)
  griddep_wait();

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------------- producer
      uint32_t na = 0, nt = 0, i = 0;
      const int count = *p.n_items;
      const int n_rt_items = p.n_rt_items;
      int item = atomicAdd(p.queue, 1);
      bool ok = true;
      while (ok && item < count) {
        const int next = atomicAdd(p.queue, 1);
        // decode the item: router items first, then tile items (tile-major)
        int kind, rt, tile, plane = 0;
        if (item < n_rt_items) {
          kind = kItemRT;
          plane = item / (p.n_rt_router * p.n_router_tiles);
          const int rem = item % (p.n_rt_router * p.n_router_tiles);
          tile = rem / p.n_rt_router;
          rt = rem % p.n_rt_router;
        } else {
          kind = p.tile_kind;
          tile = p.tile0 + (item - n_rt_items) / p.n_rt_tile;
          rt = (item - n_rt_items) % p.n_rt_tile;
        }
        const LtTile tl = p.tiles[tile];
        const uint8_t* A;
        const uint8_t* B;
        int fmt, K;
        if (kind == kItemGU) {
          fmt = tl.e >= 0 ? p.fmt : p.sfmt;
          K = p.H;
          A = (tl.e >= 0 ? p.gu + (int64_t)tl.e * p.gu_stride : p.sgu) + rt * lt_tile_bytes(fmt, K);
          B = p.xg + (int64_t)tl.prow0 * p.H * 2;
        } else if (kind == kItemDN) {
          fmt = tl.e >= 0 ? p.fmt : p.sfmt;
          K = tl.e >= 0 ? p.I : p.Ish;
          A = (tl.e >= 0 ? p.dn + (int64_t)tl.e * p.dn_stride : p.sdn) + rt * lt_tile_bytes(fmt, K);
          B = p.h + (int64_t)tl.prow0 * p.Imax * 2;
        } else {
          fmt = MOE_BF16;
          K = p.H;
          A = p.router + plane * p.router_plane + rt * lt_tile_bytes(MOE_BF16, K);
          B = p.xg + (int64_t)tl.prow0 * p.H * 2;
        }
        // item information for the epilogue
        const uint32_t j = i & 3;
        if (i >= 4 && !(ok = wait1(&iempty[j], ((i >> 2) - 1) & 1, abort, p, kSiteItem, (int)i))) break;
        infos[j] = ItemInfo{0, kind, rt, tl.e, tl.slot0, tl.n, tl.n_pad, tl.prow0, plane, {0, 0, 0}};
        mbar_arrive(&ifull[j]);
        const int span = fmt == MOE_Q8_0 ? kStageK : (fmt == MOE_Q4KS ? 256 : 128);  // columns per A stage
        const int nst = (K + span - 1) / span;
        for (int st = 0; st < nst; ++st, ++na) {
          const int c0 = st * span, cols = min(span, K - c0);
          const uint32_t sa = na % kNA;
          if (na >= kNA && !(ok = wait1(&aempty[sa], ((na / kNA) - 1) & 1, abort, p, kSiteFree, (int)na))) break;
          const int nts = 1;
          StageDesc d;
          d.flags = 0;
          d.fmt = fmt;
          d.n_pad = tl.n_pad;
          d.cols = cols;
          d.nt0 = (int)nt;
          d.nts = nts;
          d.tflags[0] = (st == 0 ? kFlagFirst : 0) | (st == nst - 1 && nts == 1 ? kFlagLast : 0);
          d.tflags[1] = st == nst - 1 ? kFlagLast : 0;
          descs[sa] = d;
          uint32_t abytes;
          const uint8_t* asrc;
          if (fmt == MOE_Q8_0) {
            asrc = A + (int64_t)(c0 / 64) * kLtQ8Chunk;
            abytes = (uint32_t)(cols / 64) * kLtQ8Chunk;
          } else if (fmt == MOE_Q4KS) {
            asrc = A + (int64_t)(c0 / 256) * kLtQ4Super;
            abytes = kLtQ4Super;
          } else {
            asrc = A + (int64_t)(c0 / 64) * kLtBf16Chunk;
            abytes = (uint32_t)(cols / 64) * kLtBf16Chunk;
          }
          mbar_arrive_expect_tx(&afull[sa], abytes);
          bulk_g2s(sm + sa * kASlot, asrc, abytes, &afull[sa]);
          // activation K-slices, one per TMEM stage
          for (int t = 0; t < nts; ++t, ++nt) {
            const int tc0 = c0 + kStageK * t, tcols = min(kStageK, cols - kStageK * t);
            // slot nt % kNB is free once the MMAs of TMEM stage nt - kNB completed
            const uint32_t sb = nt % kNB;
            if (nt >= kNB && !(ok = wait1(&tempty[sb], ((nt / kNB) - 1) & 1, abort, p, kSiteFree, -(int)nt)))
              break;
            const uint32_t bbytes = (uint32_t)tl.n_pad * tcols * 2;
            mbar_arrive_expect_tx(&bfull[sb], bbytes);
            bulk_g2s(sm + kOffB + sb * kBSlot, B + (int64_t)(tc0 / 64) * tl.n_pad * 128, bbytes, &bfull[sb]);
          }
          if (!ok) break;
        }
        ++i;
        item = next;
      }
      // end marker: one A stage, which both dequant groups see and forward
      // to the MMA issuer
      if (ok) {
        const uint32_t j = i & 3;
        if (i < 4 || (ok = wait1(&iempty[j], ((i >> 2) - 1) & 1, abort, p, kSiteItem, (int)i))) {
          infos[j].end = 1;
          mbar_arrive(&ifull[j]);
        }
      }
      for (int e = 0; e < 1 && ok; ++e, ++na) {
        const uint32_t sa = na % kNA;
        if (na >= kNA && !(ok = wait1(&aempty[sa], ((na / kNA) - 1) & 1, abort, p, kSiteFree, (int)na))) break;
        descs[sa].flags = kFlagEnd | (e == 0 ? kFlagFwdEnd : 0);
        descs[sa].nt0 = (int)nt;
        mbar_arrive(&afull[sa]);
      }
      // every copy this thread issued has landed before the CTA leaves
      const uint32_t a0 = na > kNA ? na - kNA : 0;
      for (uint32_t m = a0; m < na; ++m) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&afull[m % kNA], (m / kNA) & 1)) {
          if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_timeout(p.status, kSiteDrain, (int)m);
            break;
          }
        }
      }
      const uint32_t b0 = nt > kNB ? nt - kNB : 0;
      for (uint32_t m = b0; m < nt; ++m) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bfull[m % kNB], (m / kNB) & 1)) {
          if (globaltimer_ns() - t0 > p.timeout_ns) {
            record_timeout(p.status, kSiteDrain, -(int)m);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------------- MMA issuer
      // One thread issues every MMA of the CTA, and an MMA of N <= 64 takes
      // the tensor core only ~45 cycles: the loop keeps its ring positions
      // and phases as running counters (no divisions), steps the shared-
      // memory descriptor by adding to its address field, and unrolls the
      // usual 16 K-steps of a TMEM stage.
      uint32_t i = 0, a = 0;
      uint32_t st = 0, tph = 0, sb = 0;
      for (uint32_t nt = 0;; ++nt) {
        if (!wait1(&tfull[st], tph, abort, p, kSiteDq, (int)nt)) break;
        const TDesc d = tdescs[st];
        if (d.flags & kFlagEnd) break;
        if (d.flags & kFlagFirst) {
          a = i & 1;
          const uint32_t u = i >> 1;
          if (u >= 1 && !wait1(&dempty[a], (u - 1) & 1, abort, p, kSiteAcc, (int)i)) break;
        }
        // (the activation slot's copy was observed complete before the stage's
        // barrier, by the dequant warp that writes the stage descriptor)
        tc::fence_after();
        const uint32_t idesc = tc::idesc_f16(kLtRows, d.n_pad);
        const uint32_t lbo = (uint32_t)d.n_pad * 16;
        // K step of 16 = two core matrices along K: the address field (bits
        // 0-13, address / 16; shared addresses stay below 2^18) grows by 2 lbo / 16
        const uint64_t bdesc = tc::smem_desc(smem_u32(sm + kOffB + sb * kBSlot), lbo, 128);
        const uint64_t bstep = (uint64_t)(lbo >> 3);
        const uint32_t dacc = tbase + kTmemAcc + 64 * a, at = tbase + kTmemStage * st;
        const uint32_t acc0 = (d.flags & kFlagFirst) ? 0u : 1u;
        if (d.nk == 16) {
#pragma unroll
          for (int j = 0; j < 16; ++j) tc::mma_ts(dacc, at + 8 * j, bdesc + j * bstep, idesc, j == 0 ? acc0 : 1u);
        } else {
          for (int j = 0; j < d.nk; ++j) tc::mma_ts(dacc, at + 8 * j, bdesc + j * bstep, idesc, j == 0 ? acc0 : 1u);
        }
        tc::commit(&tempty[st]);  // frees TMEM stage st and activation slot sb (== st)
        if (d.flags & kFlagLast) {
          tc::commit(&dfull[a]);
          ++i;
        }
        if (++st == kNT) { st = 0; tph ^= 1u; }
        if (++sb == kNB) sb = 0;
      }
      // all MMAs of this thread complete before the accumulators are freed
      tc::commit(finbar);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(finbar, 0)) {
        if (globaltimer_ns() - t0 > p.timeout_ns) {
          record_timeout(p.status, kSiteDrain, -1);
          break;
        }
      }
    }
  } else if (warp >= kDequantWarp0 && warp < kEpiWarp0) {
    // ------------------------------------------------------------------ dequantise
    const int q = warp & 3, g = (warp - kDequantWarp0) >> 2, r = 32 * q + lane;
    const bool leader = warp == kDequantWarp0 && lane == 0;  // writes the TMEM stage's descriptor
    const uint32_t tlane = (uint32_t)(32 * q) << 16;
    for (uint32_t na = 0;; ++na) {
      const uint32_t sa = na % kNA;
      if (!waitw(&afull[sa], (na / kNA) & 1, abort, p, kSiteFull, (int)na)) break;
      const StageDesc d = descs[sa];
      const uint8_t* s = sm + sa * kASlot;
      const uint32_t t = (uint32_t)d.nt0, ts = t % kNT;
      if (d.flags & kFlagEnd) {
        if (d.flags & kFlagFwdEnd) {
          if (t >= kNT && !waitw(&tempty[ts], ((t / kNT) - 1) & 1, abort, p, kSiteFree, (int)t)) break;
          if (leader) tdescs[ts] = TDesc{kFlagEnd, 0, 0, 0};
          __syncwarp();
          if (lane == 0) mbar_arrive(&tfull[ts]);
        }
        break;
      }
      int nk = 0;
      if (d.fmt == MOE_Q8_0) {
        // up to 8 blocks (four 64-column K-blocks x two halves); group g
        // takes blocks 4g .. 4g+3
        const int nb = d.cols / 32;
        uint4 c[4][2];
        uint32_t sc[4];
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int b = 4 * g + bb;
          if (b < nb) {
            const uint8_t* kbp = s + (b >> 1) * kLtQ8Chunk;
            const int h = b & 1;
            c[bb][0] = *reinterpret_cast<const uint4*>(kbp + ((h * 2 + 0) * 128 + r) * 16);
            c[bb][1] = *reinterpret_cast<const uint4*>(kbp + ((h * 2 + 1) * 128 + r) * 16);
            const uint32_t h16 = *reinterpret_cast<const unsigned short*>(kbp + 8192 + (h * 128 + r) * 2);
            sc[bb] = h16 | (h16 << 16);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[sa]);
        if (t >= kNT && !waitw(&tempty[ts], ((t / kNT) - 1) & 1, abort, p, kSiteFree, (int)t)) break;
        tc::fence_after();
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int b = 4 * g + bb;
          if (b < nb) {
            uint32_t v[16];
            dq_q8(c[bb][0], c[bb][1], sc[bb], v);
            tc::st_32x32b_x16(tbase + tlane + kTmemStage * ts + 16 * b, v);
          }
        }
        nk = nb * 2;
      } else if (d.fmt == MOE_Q4KS) {
        // one superblock: header, then its 8 sub-blocks; group g takes
        // sub-blocks 4g .. 4g+3
        const uint4 hv = *reinterpret_cast<const uint4*>(s + r * 16);
        uint4 c[4];
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int sb = 4 * g + k4;
          c[k4] = *reinterpret_cast<const uint4*>(s + kLtQ4Hdr + (sb >> 1) * kLtQ4Codes + ((sb & 1) * 128 + r) * 16);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[sa]);
        const float dd = __half2float(__ushort_as_half((unsigned short)(hv.x & 0xFFFFu)));
        const float dm = __half2float(__ushort_as_half((unsigned short)(hv.x >> 16)));
        if (t >= kNT && !waitw(&tempty[ts], ((t / kNT) - 1) & 1, abort, p, kSiteFree, (int)t)) break;
        tc::fence_after();
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int sb = 4 * g + k4;
          uint32_t v[16];
          dq_q4(c[k4], dd * (float)q4_field(hv.y, hv.z, hv.w, sb), dm * (float)q4_field(hv.y, hv.z, hv.w, 8 + sb), v);
          tc::st_32x32b_x16(tbase + tlane + kTmemStage * ts + 16 * sb, v);
        }
        nk = 16;
      } else {
        // router plane: up to 128 columns of fp16 (two 64-column K-blocks),
        // copied as they are; group g takes K-block g
        const int nkb = d.cols / 64;
        uint32_t v[2][16];
        if (g < nkb) {
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) {
              const uint4 x = *reinterpret_cast<const uint4*>(s + g * kLtBf16Chunk + ((h * 4 + pc) * 128 + r) * 16);
              v[h][4 * pc + 0] = x.x;
              v[h][4 * pc + 1] = x.y;
              v[h][4 * pc + 2] = x.z;
              v[h][4 * pc + 3] = x.w;
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&aempty[sa]);
        if (t >= kNT && !waitw(&tempty[ts], ((t / kNT) - 1) & 1, abort, p, kSiteFree, (int)t)) break;
        tc::fence_after();
        if (g < nkb) {
          tc::st_32x32b_x16(tbase + tlane + kTmemStage * ts + 32 * g, v[0]);
          tc::st_32x32b_x16(tbase + tlane + kTmemStage * ts + 32 * g + 16, v[1]);
        }
        nk = nkb * 4;
      }
      tc::wait_st();
      tc::fence_before();
      bool bok = true;
      if (leader) {
        // the stage's activation slot (slot ts of the B ring) has landed: the
        // issuer then waits on this stage's barrier alone
        bok = wait1(&bfull[ts], (t / kNB) & 1, abort, p, kSiteFull, (int)t);
        tdescs[ts] = TDesc{d.tflags[0], d.n_pad, nk, 0};
      }
      if (!__shfl_sync(0xffffffffu, (int)bok, 0)) break;
      if (lane == 0) mbar_arrive(&tfull[ts]);
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp & 3, r = 32 * q + lane;
    uint8_t* stg = sm + kOffStaging + q * 2048;
    for (uint32_t i = 0;; ++i) {
      const uint32_t j = i & 3;
      if (!waitw(&ifull[j], (i >> 2) & 1, abort, p, kSiteItem, (int)i, 0)) break;
      const ItemInfo info = infos[j];
      if (info.end) break;
      const uint32_t a = i & 1;
      if (!waitw(&dfull[a], (i >> 1) & 1, abort, p, kSiteAcc, (int)i, 0)) break;
      tc::fence_after();
      const uint32_t tacc = tbase + ((uint32_t)(32 * q) << 16) + kTmemAcc + 64 * a;
      for (int c = 0; c < info.n_pad; c += 16) {
        uint32_t v[16];
        tc::ld_32x32b_x16(tacc + c, v);
        tc::wait_ld();
        if (info.kind == kItemGU) {
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const float gt = __uint_as_float(v[m]);
            const float u = __shfl_down_sync(0xffffffffu, gt, 16);
            if (lane < 16) {
              const float hv = gt / (1.f + expf(-gt)) * u;
              *reinterpret_cast<__half*>(stg + ((lane >> 3) * info.n_pad + c + m) * 16 + (lane & 7) * 2) =
                  __float2half_rn(hv);
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
  return launch_pdl(lt_gemm_kernel, grid, kGemmThreads, kSmemBytes, st, p);
}

}  // namespace moe
