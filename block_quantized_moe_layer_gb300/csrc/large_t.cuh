// large_t.cuh -- data layouts and parameters of the prefill-sized (T > 8) path.
//
// Weights get a second device copy in the "LT" layout, built at create when
// T_max > 8.  A matrix [rows, K] is cut into row tiles of 128 rows (one MMA
// M) and K-blocks of 64 columns (one pipeline stage).  For gate/up, row tile
// rt holds the 64 SwiGLU outputs o in [64 rt, 64 rt + 64): tile row
// r = 32 q + i is gate row 64 rt + 16 q + i for i < 16 and up row
// 64 rt + 16 q + i - 16 otherwise, so each 32-lane quarter of the
// accumulator holds matching gate and up rows.  For down, tile row r is
// output row 128 rt + r.
//   Q8_0 : per (tile, K-block) 8704 bytes: codes [half h][piece p][128 rows][16 B]
//          (half h = Q8_0 block 2 kb + h, piece p = its weights 16p..16p+15;
//          each code byte with its sign bit flipped, q + 128), then fp16
//          scales [h][128 rows].
//   Q4KS : per (tile, 256-column superblock) 18432 bytes: the serialised
//          16-byte headers [128 rows][16 B], then for each of its 4 K-blocks
//          codes [h][128 rows][16 B] (sub-block 2j + h, serialised nibble order).
//   16-bit (tag MOE_BF16): per (tile, K-block) 16384 bytes: [h][piece p of 8]
//          [128 rows][16 B] (the router's three fp16 planes).
// Activations that feed the MMA as its B operand (the gathered x of a token
// tile and the SwiGLU outputs h) are stored per token tile as K-blocks of
// [8 column chunks][n_pad rows][8 fp16]: one contiguous block of
// n_pad * 128 bytes per K-block, which is the operand's shared-memory image
// (8x8 core matrices, K-major, no swizzle).
#pragma once
#include "layer.cuh"

namespace moe {

constexpr int kLtRows = 128;       // MMA M: weight rows per tile
constexpr int kLtKb = 64;          // K columns per pipeline stage
constexpr int kLtMaxN = 64;        // tokens per token tile
constexpr int kLtQ8Chunk = 8704;   // 128 rows x 64 columns of Q8_0
constexpr int kLtQ4Super = 18432;  // 128 rows x 256 columns of Q4KS
constexpr int kLtQ4Hdr = 2048;
constexpr int kLtQ4Codes = 4096;
constexpr int kLtBf16Chunk = 16384;
constexpr int kLtPlanes = 3;       // router: W = W1 + 2^-11 W2 + 2^-22 W3, each fp16

enum { kItemGU = 0, kItemDN = 1, kItemRT = 2 };

// A token tile: up to 64 slots of one group (an expert, or e = -1 for the
// shared expert) that share the weights of every work item on the tile.
struct LtTile {
  int e;      // routed expert, or -1 (shared expert / plain token tile)
  int slot0;  // first slot: routed slots are positions in perm[], shared slot of token t is T*k + t
  int n;      // slots in the tile
  int n_pad;  // n rounded up to 16 (the MMA N)
  int prow0;  // first padded row of the tile in the gathered-activation buffers
  int pad[3];
};

__host__ __device__ inline int64_t lt_tile_bytes(int fmt, int K) {
  return fmt == MOE_Q8_0 ? (int64_t)136 * K : fmt == MOE_Q4KS ? (int64_t)72 * K : (int64_t)256 * K;
}

// A work item of the grouped GEMM is one 128-row weight tile against one
// token tile.  A launch's items are numbered: first n_rt_items router items
// (plane-major, then token tile, then row tile), then tile items (token tile
// tile0 + i / n_rt_tile, row tile i % n_rt_tile, of kind tile_kind).
struct LtGemmParams {
  const int* n_items;  // device: item count of the launch
  int n_rt_items, n_rt_router, n_router_tiles;
  int tile_kind, tile0, n_rt_tile;
  int* queue;
  int* exit_cnt;
  int* status;
  const LtTile* tiles;
  const uint8_t* gu;
  const uint8_t* dn;
  const uint8_t* sgu;
  const uint8_t* sdn;
  const uint8_t* router;
  int64_t gu_stride, dn_stride, router_plane;
  int fmt, sfmt;
  int H, I, Ish, Imax, E_pad128, T, k;
  const uint8_t* xg;  // B of gate/up and router items
  uint8_t* h;         // gate/up output, B of down items
  __nv_bfloat16* z;   // down output [T*k + T][H]
  float* logits;      // router output [planes][T][E_pad128]
  uint64_t timeout_ns;
};

cudaError_t lt_gemm_configure();
cudaError_t lt_gemm_launch(const LtGemmParams& p, int grid, cudaStream_t st);

}  // namespace moe
