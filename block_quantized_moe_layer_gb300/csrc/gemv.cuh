// gemv.cuh -- the integer block dot products of the T <= 8 GEMV (the MoE
// layer's expert tiles and the LM head).
//
// A weight chunk holds 32 rows (lane = row) x Kc columns in the streaming
// chunk layout (common.cuh, chunk_bytes); the activations of the M vectors
// are block fixed-point records (common.cuh, write_record), laid out
// [M][nbc] right after the chunk's data in shared memory or anywhere else.
// Weights enter as their integer codes, activations as L-limb block fixed
// point; dp4a gives exact integer block sums, scaled once per block:
//   Q8_0 : sum_i d q_i v_i       = d * ascale * sum_i q_i X_i
//   Q4KS : sum_i (a q_i - b) v_i = a * ascale * sum_i q_i X_i - b * sumx
#pragma once
#include "common.cuh"

namespace moe {

// Integer dot product of one 32-weight Q8_0 block (codes q0 | q1) with one
// activation record: four independent dp4a chains of four, then the limbs
// combined exactly (L = 2) or in fp32 (L = 4).
template <int L>
__device__ __forceinline__ float q8_block(const uint4 q0, const uint4 q1, const uint8_t* rec) {
  int c[2 * L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(rec + 32 * l);
    const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 32 * l + 16);
    if (l == L - 1) {  // top limb: signed
      c[2 * l] = dp4a_ss(q0.w, a0.w, dp4a_ss(q0.z, a0.z, dp4a_ss(q0.y, a0.y, dp4a_ss(q0.x, a0.x, 0))));
      c[2 * l + 1] = dp4a_ss(q1.w, a1.w, dp4a_ss(q1.z, a1.z, dp4a_ss(q1.y, a1.y, dp4a_ss(q1.x, a1.x, 0))));
    } else {
      c[2 * l] = dp4a_su(q0.w, a0.w, dp4a_su(q0.z, a0.z, dp4a_su(q0.y, a0.y, dp4a_su(q0.x, a0.x, 0))));
      c[2 * l + 1] = dp4a_su(q1.w, a1.w, dp4a_su(q1.z, a1.z, dp4a_su(q1.y, a1.y, dp4a_su(q1.x, a1.x, 0))));
    }
  }
  if constexpr (L == 2) {
    return (float)((c[2] + c[3]) * 256 + (c[0] + c[1]));
  } else {
    return fmaf((float)(c[6] + c[7]), 16777216.f,
                fmaf((float)(c[4] + c[5]), 65536.f, fmaf((float)(c[2] + c[3]), 256.f, (float)(c[0] + c[1]))));
  }
}

// Same for one 32-weight Q4KS sub-block held as 16 bytes of codes (qv): the
// low nibbles of word j are codes 8j..8j+3, the high nibbles codes
// 8j+4..8j+7.  The high nibbles stay in place, so their products come out
// 16 times too large; each such sum is a multiple of 16 and is divided back
// exactly (an arithmetic shift, which the CUDA compiler guarantees for
// signed integers).
template <int L>
__device__ __forceinline__ float q4_block(const uint4 qv, const uint8_t* rec) {
  const uint32_t l0 = qv.x & 0x0F0F0F0Fu, l1 = qv.y & 0x0F0F0F0Fu, l2 = qv.z & 0x0F0F0F0Fu, l3 = qv.w & 0x0F0F0F0Fu;
  const uint32_t h0 = qv.x & 0xF0F0F0F0u, h1 = qv.y & 0xF0F0F0F0u, h2 = qv.z & 0xF0F0F0F0u, h3 = qv.w & 0xF0F0F0F0u;
  int lo[L], hi[L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(rec + 32 * l);
    const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 32 * l + 16);
    if (l == L - 1) {  // top limb: signed
      lo[l] = dp4a_us(l3, a1.z, dp4a_us(l2, a1.x, dp4a_us(l1, a0.z, dp4a_us(l0, a0.x, 0))));
      hi[l] = dp4a_us(h3, a1.w, dp4a_us(h2, a1.y, dp4a_us(h1, a0.w, dp4a_us(h0, a0.y, 0))));
    } else {
      lo[l] = dp4a_uu(l3, a1.z, dp4a_uu(l2, a1.x, dp4a_uu(l1, a0.z, dp4a_uu(l0, a0.x, 0))));
      hi[l] = dp4a_uu(h3, a1.w, dp4a_uu(h2, a1.y, dp4a_uu(h1, a0.w, dp4a_uu(h0, a0.y, 0))));
    }
  }
  if constexpr (L == 2) {
    // lo0 + 256 lo1 + (hi0 + 256 hi1) / 16, all terms exact in int32
    return (float)(lo[0] + lo[1] * 256 + hi[1] * 16 + (hi[0] >> 4));
  } else {
    const int c0 = lo[0] + (hi[0] >> 4), c1 = lo[1] + (hi[1] >> 4), c2 = lo[2] + (hi[2] >> 4),
              c3 = lo[3] + (hi[3] >> 4);
    return fmaf((float)c3, 16777216.f, fmaf((float)c2, 65536.f, fmaf((float)c1, 256.f, (float)c0)));
  }
}

// Scales of sub-block `sub` from a 16-byte superblock header (fp16 d | fp16
// dmin, then 16 six-bit fields: sc[0..7] at bits 6s, m[0..7] at 48 + 6s of
// the following 96 bits): a = d * sc, b = dmin * m, exact in fp32 (11 x 6
// significant bits).  2^23 + v is the float with bits 0x4B000000 | v, and
// one fma with -d * 2^23 removes the 2^23 term with a single exact rounding.
// `sub` is the same for a warp over a whole chunk, so the shifts and word
// choices are loop constants.
__device__ __forceinline__ void q4_scales(const uint4 hd, int sub, float dd, float dmin, float& a, float& b) {
  const uint32_t sh_sc = (uint32_t)(6 * sub) & 31u, sh_m = (uint32_t)(48 + 6 * sub) & 31u;
  const bool sc_low = sub <= 5, m_low = sub <= 2;  // field starts in the first word of its pair
  const uint32_t sc = __funnelshift_r(sc_low ? hd.y : hd.z, sc_low ? hd.z : hd.w, sh_sc) & 63u;
  const uint32_t mm = __funnelshift_r(m_low ? hd.z : hd.w, m_low ? hd.w : 0u, sh_m) & 63u;
  a = fmaf(dd, __uint_as_float(0x4B000000u | sc), -dd * 8388608.f);
  b = fmaf(dmin, __uint_as_float(0x4B000000u | mm), -dmin * 8388608.f);
}

// One chunk.  Lane l owns row l of the chunk; warp w owns blocks w, w + 8,
// ... (a warp load of one block's 16-byte pieces covers the 32 rows in 512
// contiguous bytes; the block's activation records are a broadcast read, one
// per warp).  acc[m] collects this warp's share of the lane's row against
// vector m; the 8 warps' shares are summed by the epilogue warp.
template <int L, int M>
__device__ __forceinline__ void gemv_chunk_m(const uint8_t* stage, const uint8_t* A, int nbc, int fmt, int group,
                                             float (&acc)[kGroup]) {
  constexpr int RB = rec_bytes(L);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (fmt == MOE_Q8_0) {
    const __half* sc = reinterpret_cast<const __half*>(stage + nbc * 1024);
#pragma unroll 2
    for (int b = warp; b < nbc; b += kBlocksPerStep) {
      const uint4 q0 = *reinterpret_cast<const uint4*>(stage + ((int64_t)(b * 2 + 0) * kRows + lane) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(stage + ((int64_t)(b * 2 + 1) * kRows + lane) * 16);
      const float dq = __half2float(sc[b * kRows + lane]);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint8_t* rec = A + (m * nbc + b) * RB;
        const float asc = *reinterpret_cast<const float*>(rec + 32 * L);
        acc[m] = fmaf(dq * asc, q8_block<L>(q0, q1, rec), acc[m]);
      }
    }
  } else {  // MOE_Q4KS
    // Pairs of blocks (2i, 2i+1) of the group; the pairs of a stage's groups,
    // numbered group * nbc/2 + i, go round robin to the 8 warps.  A chunk is
    // whole 256-column superblocks (4 pairs), so a warp's pairs always sit at
    // the same place in their superblock: sub-blocks s0 and s0 + 1, whose
    // header it reads once for both.
    static_assert(kBlocksPerStep == 8, "8 warps share a stage");
    const uint8_t* hdr = stage + nbc * 512;
    const int np = nbc >> 1;
    const int p0 = (warp - group * np) & 7;
    const int s0 = (2 * p0) & 7;
#pragma unroll 2
    for (int p = p0; p < np; p += kBlocksPerStep) {
      const int b = 2 * p;
      const uint4 hd = *reinterpret_cast<const uint4*>(hdr + ((b >> 3) * kRows + lane) * 16);
      const float dd = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
      const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const uint4 qv = *reinterpret_cast<const uint4*>(stage + ((int64_t)(b + i) * kRows + lane) * 16);
        float sa, sb;
        q4_scales(hd, s0 + i, dd, dmin, sa, sb);
#pragma unroll
        for (int m = 0; m < M; ++m) {
          const uint8_t* rec = A + (m * nbc + b + i) * RB;
          const float asc = reinterpret_cast<const float*>(rec + 32 * L)[0];
          const float sx = reinterpret_cast<const float*>(rec + 32 * L)[1];
          acc[m] = fmaf(sa * asc, q4_block<L>(qv, rec), fmaf(-sb, sx, acc[m]));
        }
      }
    }
  }
}

// The token count of a stage as a compile-time constant, so the loops over
// tokens unroll without predicates (a runtime bound there keeps the loads of
// different tokens from being scheduled together).
template <int L>
__device__ __forceinline__ void gemv_chunk(const uint8_t* stage, const uint8_t* A, int nbc, int fmt, int group, int M,
                                           float (&acc)[kGroup]) {
  switch (M) {
    case 1: gemv_chunk_m<L, 1>(stage, A, nbc, fmt, group, acc); break;
    case 2: gemv_chunk_m<L, 2>(stage, A, nbc, fmt, group, acc); break;
    case 3: gemv_chunk_m<L, 3>(stage, A, nbc, fmt, group, acc); break;
    default: gemv_chunk_m<L, kGroup>(stage, A, nbc, fmt, group, acc); break;
  }
}

}  // namespace moe
