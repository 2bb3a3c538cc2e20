// A TMA-fed tcgen05 GEMM engine for the DyRA forward: D[b] = A[b] B[b]^T with both operands
// stored K-contiguous ("K-major") or MN-contiguous, fp32 accumulation in TMEM.
//
// Persistent kernel: a grid of at most one CTA per SM walks the tiles (batch, m tile,
// n tile), n fastest, in a static round-robin. In pair-MMA mode (cta_group::2) a 2-CTA
// cluster takes adjacent M tiles of one (batch, N tile) as a 256-row unit: each CTA loads its
// own 128 rows of A and its own half of the B tile into its own shared memory, the even CTA
// issues the MMAs for both, and each CTA's TMEM receives its own 128 rows.
// Each CTA has these warps:
//   warp 0      TMA issuer for A (one lane): 128-byte K chunks (128 rows) into a ring of
//               shared-memory stages; it runs ahead across tile boundaries
//   warp 1      TMEM allocation and MMA issue (one lane): 4 MMAs (32 bytes of K each) per
//               chunk into one of two TMEM accumulators, so the epilogue of tile i overlaps
//               the main loop of tile i+1
//   warp 2      TMA issuer for B (one lane)
//   warps 4..11 epilogue, two warps per TMEM lane quarter (each a column half): tcgen05.ld
//               of the accumulator (one row per thread), then the epilogue mode below;
//               row-major bf16 results go through 64-byte-swizzled shared-memory staging
//               tiles and TMA bulk stores
// Operands are bf16 (kind::f16, K-major or MN-major) or fp32 read as tf32 (kind::tf32,
// K-major only), always in the 128-byte swizzled layout that TMA writes. The B operand
// may switch major-ness at the K chunk b_split (e.g. a K-major weight followed by an
// MN-major per-sample factor). In segmented mode (seg_n) the M rows are the flat rows of
// several samples and the chunks from b_split on repeat once per sample a unit touches.
//
// The issuing threads run short dependent instruction chains, so their loops keep
// everything precomputed: shared-memory descriptors are built once and advanced by adding
// to their address field, the ring position advances by increment and wrap, and no
// division happens inside the K loop.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

namespace dyra {

enum TcEpi : int {
  EPI_ROW_BF16 = 0,    // out[b][g][c] = bf16(acc + bias[c]); TMA store when tma_store is set
  EPI_CG = 2,          // m tiles < a_split: out[b*bs + g*ld + c] = acc     (C^T, fp32)
                       // m tiles >= a_split: out2[b*bs2 + g*ld2 + c] = acc  (G, fp32)
  EPI_ROW_F32 = 3,     // m tiles < a_split: out[b][g][c] = alpha*acc + beta*aux[b][g][c]
                       // m tiles >= a_split: out2[b][g][c] = alpha*acc + beta*aux2[b][g][c]
                       // (fp32; aux / aux2 may be null; 16-byte vector accesses)
  EPI_CG_SOLVE = 5     // the Gram GEMM [X | L]^T L with the r <= 64 SPD solve folded in: the
                       // G tile of a sample (walked first) is inverted by the epilogue warps
                       // (block sweeps, solve_r <= 64) and published (ginv32 / ginv16, then
                       // ready[b] = 1); a C^T tile waits for its sample's G^-1 and
                       // writes C^T (out, fp32) and C~ = G^-1 C (cs [b][r][d], bf16)
};

struct TcGemmParams {
  int m_tiles, n_tiles, batch;
  int pair_mma;      // 1: CTA pairs run cta_group::2 MMAs (M = 256 per pair): each CTA holds
                     // its 128 rows of A and half of the B tile (BN / 2 rows or columns), the
                     // even CTA issues the MMAs, each CTA's TMEM receives its own 128 rows
                     // (K-major B maps then need a box of BN / 2 rows; MN-major B needs
                     // BN % 128 == 0)
  int cluster;       // set by tc_gemm_launch: 2 with pair_mma, else 1
  int BN;            // MMA N of a tile: multiple of 16 (of 64 for MN-major B), <= 256
  int k_chunks;      // K in 128-byte chunks
  int elem_bytes;    // 2 = bf16, 4 = fp32/tf32
  int a_major, b_major;   // 0 = K-major, 1 = MN-major
  int a_split;       // m tiles >= a_split load from map A1 (M coordinate restarts at 0)
  int a_batched0, a_batched1;  // map carries the batch coordinate
  int b_split;       // k chunks >= b_split load from map B1 (K coordinate restarts at 0)
  int b_batched0, b_batched1;
  int b_major1;      // major of the chunks read from map B1
  int a_kdiag;       // > 0: K-major A chunks < b_split are read at K = n_tile * a_kdiag +
                     // kc * chunk (block-diagonal B: N tile j only contracts with its own
                     // a_kdiag-wide range of K; Monarch: a_kdiag = BN)
  int a_k1;          // K coordinate of A (elements) read by chunk b_split; later chunks follow
                     // it. < 0: contiguous with the chunks before (b_split * chunk)
  int seg_n;         // > 0: flat M over `seg_count` segments (samples) of seg_n rows each.
                     // Chunks >= b_split then repeat once per segment that the rows of the
                     // tile (of the CTA pair, for pair MMAs) touch: A from map A1 as
                     // [segment][seg_n][inner] at row (first row of the tile - segment start),
                     // whose rows outside the segment read as zeros, and B from map B1 with
                     // the segment as its batch coordinate. Needs batch = 1, K-major A.
  int seg_count;
  uint32_t idesc;
  uint32_t idesc1;   // instruction descriptor of the chunks read from map B1
  uint32_t acc_cols;  // TMEM columns of one accumulator (power of two >= BN)
  int stages;
  uint32_t smem_bytes;
  uint32_t staging_off;  // byte offset of the epilogue staging buffers (TMA store)
  uint32_t bar_off;      // byte offset of the mbarriers (after the staging buffers)
  // epilogue
  int epi;
  int tma_store;     // EPI_ROW_BF16 through the output tensor map (needs BN % 32 == 0)
  int epi_bufs;      // staging-tile pairs per epilogue warp (1 or 2; 0: chosen at launch)
  int act;           // TMA-store epilogue: 0 none, 1 GELU (erf form) after the bias
  int out_batched;   // output map carries the batch coordinate
  void *out;
  long long out_bstride, out_ld;
  int rows_valid, cols_valid;     // region of tiles < a_split
  void *out2;
  long long out2_bstride, out2_ld;
  int rows2_valid, cols2_valid;   // region of tiles >= a_split (EPI_CG, EPI_ROW_F32)
  const float *bias;
  const float *aux, *aux2;        // addends of EPI_ROW_F32's two regions (or null)
  long long aux_bstride, aux_ld, aux2_bstride, aux2_ld;
  float alpha, beta;
  int *timeouts;                  // device counter of bounded waits that gave up
  int m_fast;                     // walk M tiles fastest (a large B shared by few M tiles:
                                  // the units running together read the same B columns)
  // EPI_CG_SOLVE
  int g_first;                    // the walk takes every sample's G tile first
  int solve_r;                    // r (<= 64, % 4 == 0)
  float ridge;
  float *ginv32;                  // [batch][r][r] fp32 (G + ridge I)^-1
  __nv_bfloat16 *ginv16;          // [batch][r][r] bf16
  __nv_bfloat16 *cs;              // [batch][r][d] bf16 C~
  int cs_d;                       // d
  int *ready;                     // [2][batch]: G^-1 of the sample published; C tiles that
                                  // have read it (the last one sets both back to 0)
  int *nspd;                      // counter of samples that are not positive definite
  uint32_t solve_off;             // shared-memory offset of the solve scratch
};

struct TcOperand {
  // One TMA source: a [batch][rows][inner] tensor (inner contiguous).
  const void *base;
  int elem_bytes;
  long long inner, rows, batch;         // extents in elements
  long long row_stride, batch_stride;   // in bytes
};

// Build the instruction descriptor (M = 128, or 256 for pair MMAs).
uint32_t tc_idesc(int elem_bytes, int a_major, int b_major, int n, int m = 128);

// Creates a 3-D tensor map with 128-byte swizzle, box = {chunk, box_rows, 1}.
bool tc_make_map(CUtensorMap *map, const TcOperand &op, int box_rows);

// Creates the bf16 output map of the TMA-store epilogue: box {32, 32, 1}, 64-byte swizzle.
bool tc_make_store_map(CUtensorMap *map, const TcOperand &op);

// Fills stages / smem / TMEM columns / grid for a given BN and launches the kernel.
// `out_map` is used only when p.tma_store is set.
cudaError_t tc_gemm_launch(TcGemmParams p, const CUtensorMap &a0, const CUtensorMap &a1,
                           const CUtensorMap &b0, const CUtensorMap &b1,
                           const CUtensorMap &out_map, cudaStream_t stream);

}  // namespace dyra
