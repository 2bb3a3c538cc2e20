// Persistent TMA + tcgen05 GEMM engine used by every dense contraction of the bf16 DyRA
// forward. See tc_gemm.cuh for the roles of the warps and the epilogue modes.
#include "tc_gemm.cuh"
#include "ptx.cuh"
#include "sweep.cuh"

#include <cuda_bf16.h>
#include <cstring>
#include <map>
#include <mutex>

namespace dyra {

namespace {

constexpr uint32_t kStagingPairBytes = 2 * 2048;   // one pair of 32 x 32 bf16 staging tiles

// GELU(x) = x Phi(x) = x (1 + erf(x / sqrt 2)) / 2 (the erf form of the ViT MLP blocks).
__device__ __forceinline__ float gelu_erf(float x) {
  return 0.5f * x * (1.f + erff(x * 0.70710678118654752f));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

struct TileCoord {
  int bz, m_tile, n_tile;
};

// Shared-memory scratch of the EPI_CG_SOLVE epilogue.
struct alignas(16) SolveSmem {
  int got, ok, pad[2];
  float Gs[64][68];        // G of a G tile, or G^-1 for a C tile (row pitch 68 floats)
  sweep::Smem<32> s32;
  sweep::Smem<64> s64;
};

// Named barrier of the 8 epilogue warps.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Unit u of the persistent walk (n fastest); with pair MMAs (cluster = 2) a unit is a pair
// of M tiles and CTA rank `crank` of the cluster takes M tile 2 * pair + crank (possibly one
// past the last M tile: then its loads read zeros and its epilogue stores nothing).
__device__ __forceinline__ TileCoord decode_tile(int u, const TcGemmParams &p, int mp_tiles,
                                                 int crank) {
  TileCoord c;
  if (p.g_first) {   // single CTAs, one N tile, m_tiles = a_split + 1: every G tile first
    c.n_tile = 0;
    if (u < p.batch) {
      c.bz = u;
      c.m_tile = p.a_split;
    } else {
      u -= p.batch;
      c.m_tile = u % p.a_split;
      c.bz = u / p.a_split;
    }
    return c;
  }
  if (p.m_fast) {
    c.m_tile = (u % mp_tiles) * p.cluster + crank;
    const int rest = u / mp_tiles;
    c.n_tile = rest % p.n_tiles;
    c.bz = rest / p.n_tiles;
    return c;
  }
  c.n_tile = u % p.n_tiles;
  const int rest = u / p.n_tiles;
  c.m_tile = (rest % mp_tiles) * p.cluster + crank;
  c.bz = rest / mp_tiles;
  return c;
}

// K chunks of the tile (segmented mode: b_split plus one group of rank chunks per segment
// that the unit's rows touch) and the first segment it touches.
__device__ __forceinline__ int tile_chunks(const TcGemmParams &p, const TileCoord &tc, int crank,
                                           int &s_lo) {
  if (p.seg_n <= 0) {
    s_lo = 0;
    return p.k_chunks;
  }
  const int urow0 = (tc.m_tile - crank) * 128;   // first row of the CTA pair's unit
  s_lo = urow0 / p.seg_n;
  int s_hi = (urow0 + 128 * p.cluster - 1) / p.seg_n;
  if (s_hi > p.seg_count - 1) s_hi = p.seg_count - 1;
  return p.b_split + (s_hi - s_lo + 1) * (p.k_chunks - p.b_split);
}

// dst[0..16) = alpha * f[0..16) + beta * ax[0..16) (ax may be null) for the first `valid`
// columns; 16-byte vector accesses when every column is valid and the rows are aligned.
__device__ __forceinline__ void store_row16_f32(float *dst, const float *ax, const float *f,
                                                int valid, float alpha, float beta) {
  if (valid >= 16 && ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(ax)) & 15) == 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float4 o = make_float4(alpha * f[4 * q], alpha * f[4 * q + 1], alpha * f[4 * q + 2],
                             alpha * f[4 * q + 3]);
      if (ax) {
        const float4 a = *reinterpret_cast<const float4 *>(ax + 4 * q);
        o.x += beta * a.x;
        o.y += beta * a.y;
        o.z += beta * a.z;
        o.w += beta * a.w;
      }
      *reinterpret_cast<float4 *>(dst + 4 * q) = o;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < valid) dst[j] = alpha * f[j] + (ax ? beta * ax[j] : 0.f);
}

// Epilogue of 16 accumulator columns [col0, col0 + 16) of row g, direct global stores
// (the modes without a TMA store: C / G of the Gram kernel, fp32 Newton-Schulz products).
__device__ __forceinline__ void epilogue16(const TcGemmParams &p, const float *f, long long g,
                                           int col0, int bz, bool second) {
  const int cols_lim = second ? p.cols2_valid : p.cols_valid;
  const int valid = cols_lim - col0;
  if (valid <= 0) return;
  if (p.epi == EPI_ROW_BF16) {
    if (g < p.rows_valid) {
      __nv_bfloat16 *dst =
          reinterpret_cast<__nv_bfloat16 *>(p.out) + bz * p.out_bstride + g * p.out_ld + col0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < valid) dst[j] = __float2bfloat16_rn(f[j] + (p.bias ? __ldg(p.bias + col0 + j) : 0.f));
    }
  } else if (!second) {   // EPI_CG (C^T) and EPI_ROW_F32, first region
    if (g < p.rows_valid) {
      float *dst = reinterpret_cast<float *>(p.out) + bz * p.out_bstride + g * p.out_ld + col0;
      const float *ax = p.aux ? p.aux + bz * p.aux_bstride + g * p.aux_ld + col0 : nullptr;
      store_row16_f32(dst, ax, f, valid, p.alpha, p.beta);
    }
  } else if (g < p.rows2_valid) {   // second region (G of the Gram kernel, X of Newton-Schulz)
    float *dst = reinterpret_cast<float *>(p.out2) + bz * p.out2_bstride + g * p.out2_ld + col0;
    const float *ax = p.aux2 ? p.aux2 + bz * p.aux2_bstride + g * p.aux2_ld + col0 : nullptr;
    store_row16_f32(dst, ax, f, valid, p.alpha, p.beta);
  }
}

// 32 fp32 accumulator values (raw bits) of one row -> bf16 into a 32 x 32 staging tile
// (64-byte rows, 64-byte swizzle: 16-byte chunk c of row l lands at chunk c ^ ((l >> 1) & 3)).
__device__ __forceinline__ void stage_bits32(uint32_t buf, int lane, const uint32_t *v) {
  const uint32_t dst = buf + (uint32_t)lane * 64u;
  const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w0 = pack_bf16x2(__uint_as_float(v[8 * c + 0]), __uint_as_float(v[8 * c + 1]));
    const uint32_t w1 = pack_bf16x2(__uint_as_float(v[8 * c + 2]), __uint_as_float(v[8 * c + 3]));
    const uint32_t w2 = pack_bf16x2(__uint_as_float(v[8 * c + 4]), __uint_as_float(v[8 * c + 5]));
    const uint32_t w3 = pack_bf16x2(__uint_as_float(v[8 * c + 6]), __uint_as_float(v[8 * c + 7]));
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (((uint32_t)c ^ sw) << 4)),
                 "r"(w0), "r"(w1), "r"(w2), "r"(w3)
                 : "memory");
  }
}

constexpr int kWarpLoadA = 0, kWarpMma = 1, kWarpLoadB = 2;
constexpr int kEpiWarp0 = 4, kEpiWarps = 8;      // warps 4..11: two per TMEM lane quarter
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);

// C~[i][g] = sum_j G^-1[i][j] C[j][g] for rows i_lo .. i_hi - 1 of one feature g (cv = the
// feature's C column, zero past r; G^-1 rows in shared memory, zero-padded to RR columns past
// r). Each row of G^-1 is read into registers before its FMAs (the reads of one row are
// independent), and two rows go at once.
template <int RR>
__device__ __forceinline__ void apply_rows(const float (&Gs)[64][68], const float (&cv)[64],
                                           int i_lo, int i_hi, int d, __nv_bfloat16 *op) {
  constexpr int V = RR / 4;
  for (int ii = i_lo; ii < i_hi; ii += 2) {
    const bool two = ii + 1 < i_hi;
    const float4 *g0 = reinterpret_cast<const float4 *>(&Gs[ii][0]);
    const float4 *g1 = reinterpret_cast<const float4 *>(&Gs[two ? ii + 1 : ii][0]);
    float4 w0[V], w1[V];
#pragma unroll
    for (int j4 = 0; j4 < V; ++j4) {
      w0[j4] = g0[j4];
      w1[j4] = g1[j4];
    }
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f, t0 = 0.f, t1 = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
    for (int j4 = 0; j4 < V; ++j4) {
      s0 = fmaf(w0[j4].x, cv[4 * j4], s0);
      s1 = fmaf(w0[j4].y, cv[4 * j4 + 1], s1);
      s2 = fmaf(w0[j4].z, cv[4 * j4 + 2], s2);
      s3 = fmaf(w0[j4].w, cv[4 * j4 + 3], s3);
      t0 = fmaf(w1[j4].x, cv[4 * j4], t0);
      t1 = fmaf(w1[j4].y, cv[4 * j4 + 1], t1);
      t2 = fmaf(w1[j4].z, cv[4 * j4 + 2], t2);
      t3 = fmaf(w1[j4].w, cv[4 * j4 + 3], t3);
    }
    op[(size_t)ii * d] = __float2bfloat16_rn((s0 + s1) + (s2 + s3));
    if (two) op[(size_t)(ii + 1) * d] = __float2bfloat16_rn((t0 + t1) + (t2 + t3));
  }
}

// Rows i0 .. i0 + 3, columns j0 .. j0 + 3 of G^-1 (the block holds -G^-1; 0 for a sample that
// is not positive definite) to ginv32 (fp32) and ginv16 (bf16).
__device__ __forceinline__ void store_ginv_block(const TcGemmParams &p, int bz, int r, int i0,
                                                 int j0, const float (&a)[4][4], bool bad) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const size_t o = ((size_t)bz * r + i0 + u) * r + j0;
    const float4 x = bad ? make_float4(0.f, 0.f, 0.f, 0.f)
                         : make_float4(-a[u][0], -a[u][1], -a[u][2], -a[u][3]);
    *reinterpret_cast<float4 *>(p.ginv32 + o) = x;
    __nv_bfloat162 h0 = __floats2bfloat162_rn(x.x, x.y), h1 = __floats2bfloat162_rn(x.z, x.w);
    uint2 hv;
    hv.x = *reinterpret_cast<uint32_t *>(&h0);
    hv.y = *reinterpret_cast<uint32_t *>(&h1);
    *reinterpret_cast<uint2 *>(p.ginv16 + o) = hv;
  }
}

// EPI_CG_SOLVE epilogue, run by the 8 epilogue warps together (every decision is taken by one
// thread, handed out through shared memory and a named barrier, so all 8 warps meet the same
// barriers whatever a bounded wait returned).
//   G tile (rows 0..r-1 of the accumulator): G to shared memory, the accumulator released,
//     (G + ridge I)^-1 by block sweeps (sweep::invert_blocks over the 256 epilogue threads),
//     G^-1 to ginv32 / ginv16, then ready[b] = 1 (release, after a fence).
//   C^T tile (128 rows = input features g, r columns): wait until ready[b] is set (acquire,
//     bounded), stage G^-1 in shared memory, count the tile in ready[batch + b] (the last of
//     the sample's tiles clears both words for the next launch), read the tile's rows from
//     TMEM (each thread a full row), release the accumulator, write C^T (fp32) and
//     C~[b][i][g] = sum_j G^-1[i][j] C[j][g] (bf16), the two warps of a lane quarter splitting
//     the r output rows.
__device__ __noinline__ void cg_solve_epilogue(const TcGemmParams &p, uint8_t *smem, uint32_t base,
                                               uint32_t tmem_base, uint32_t tfull_bar,
                                               uint32_t tempty_bar, int cid, int ncl, int total,
                                               int mp_tiles, int e, int lane, int c_lo, int c_hi) {
  SolveSmem &ss = *reinterpret_cast<SolveSmem *>(smem + p.solve_off);
  const int et = e * 32 + lane;   // 0 .. 255 over the epilogue warps
  const int q = (kEpiWarp0 + e) & 3;
  const int r = p.solve_r, d = p.cs_d;
  uint32_t i = 0;
  for (int t = cid; t < total; t += ncl, ++i) {
    const uint32_t acc = i & 1u;
    const TileCoord tc = decode_tile(t, p, mp_tiles, 0);
    if (et == 0) ss.got = ptx::mbar_wait(tfull_bar + 8u * acc, (i >> 1) & 1u, p.timeouts) ? 1 : 0;
    epi_bar();
    const bool got = ss.got != 0;
    epi_bar();   // every warp has read ss.got before thread 0 may write it again
    if (!got) break;
    ptx::tc_fence_after();
    const uint32_t taddr = tmem_base + acc * p.acc_cols + ((uint32_t)(q * 32) << 16);
    const int bz = tc.bz;
    if (tc.m_tile >= p.a_split) {
      // ---------------------------------------------------------------- G tile
      const int row = q * 32 + lane;
      if (q * 32 < r) {   // uniform per warp: this lane quarter holds rows of G
        for (int c0 = c_lo; c0 < c_hi && c0 < r; c0 += 32) {
          uint32_t v[32];
          ptx::tmem_ld32(taddr + (uint32_t)c0, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (row < r && c0 + j < r) ss.Gs[row][c0 + j] = __uint_as_float(v[j]);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty_bar + 8u * acc);   // the accumulator is free
      epi_bar();
      if (p.out2) {   // G itself (without the ridge), kept for checks of the intermediates
        float *go = reinterpret_cast<float *>(p.out2) + (size_t)bz * r * r;
        for (int k = et; k < r * r; k += 256) go[k] = ss.Gs[k / r][k % r];
      }
      // (G + ridge I)^-1 by block sweeps over the epilogue threads (R = 32: the first 64)
      bool bad;
      float a[4][4];
      if (r <= 32) {
        const int i0 = (et / 8) * 4, j0 = (et % 8) * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int ii = i0 + u, jj = j0 + w;
            a[u][w] = (et < 64 && ii < r && jj < r) ? ss.Gs[ii][jj] + (ii == jj ? p.ridge : 0.f)
                                                    : (ii == jj ? 1.f : 0.f);
          }
        bad = !sweep::invert_blocks<32>(a, et, r, ss.s32, []() { epi_bar(); });
        if (et < 64 && i0 < r && j0 < r) store_ginv_block(p, bz, r, i0, j0, a, bad);
      } else {
        const int i0 = (et / 16) * 4, j0 = (et % 16) * 4;
#pragma unroll
        for (int u = 0; u < 4; ++u)
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const int ii = i0 + u, jj = j0 + w;
            a[u][w] = (ii < r && jj < r) ? ss.Gs[ii][jj] + (ii == jj ? p.ridge : 0.f)
                                         : (ii == jj ? 1.f : 0.f);
          }
        bad = !sweep::invert_blocks<64>(a, et, r, ss.s64, []() { epi_bar(); });
        if (i0 < r && j0 < r) store_ginv_block(p, bz, r, i0, j0, a, bad);
      }
      __threadfence();
      epi_bar();   // every thread's G^-1 stores are fenced
      if (et == 0) {   // thread 0 took part in the inversion and holds its flag
        if (bad) atomicAdd(p.nspd, 1);
        st_release_gpu(p.ready + bz, 1);
      }
    } else {
      // ---------------------------------------------------------------- C^T tile
      if (et == 0) {
        int ok = 0;
        if (ld_acquire_gpu(p.ready + bz) != 0) {
          ok = 1;
        } else {
          const unsigned long long t0 = ptx::global_timer();
          for (;;) {
            __nanosleep(200);
            if (ld_acquire_gpu(p.ready + bz) != 0) {
              ok = 1;
              break;
            }
            if (ptx::global_timer() - t0 > ptx::kWaitLimitNs) {
              atomicAdd(p.timeouts, 1);
              break;
            }
          }
        }
        ss.ok = ok;
      }
      epi_bar();
      const bool ok = ss.ok != 0;
      {   // G^-1 of the sample into shared memory (L2 reads: another CTA wrote it)
        const float *gi = p.ginv32 + (size_t)bz * r * r;
        for (int k4 = et; k4 < r * r / 4; k4 += 256) {
          const int ii = (4 * k4) / r, jj = (4 * k4) % r;
          const float4 v = ok ? __ldcg(reinterpret_cast<const float4 *>(gi) + k4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4 *>(&ss.Gs[ii][jj]) = v;
        }
        // columns r .. RR - 1 of those rows (RR = 32 or 64, what the apply reads) are zero
        const int pad = (r <= 32 ? 32 : 64) - r;
        for (int k = et; k < r * pad; k += 256) ss.Gs[k / pad][r + k % pad] = 0.f;
      }
      epi_bar();   // G^-1 is staged
      if (et == 0) {   // the last of the sample's C tiles to read G^-1 resets its flag
        if (atomicAdd(p.ready + p.batch + bz, 1) == p.a_split - 1) {
          p.ready[p.batch + bz] = 0;
          p.ready[bz] = 0;
        }
      }
      // this thread's row of C^T (input feature g), all r columns
      const int g = (tc.m_tile * 128) + q * 32 + lane;
      float cv[64];
      {
        uint32_t v[32];
        ptx::tmem_ld32(taddr, v);
        ptx::tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) cv[j] = __uint_as_float(v[j]);
        if (r > 32) {
          ptx::tmem_ld32(taddr + 32u, v);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) cv[32 + j] = __uint_as_float(v[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) cv[32 + j] = 0.f;
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(tempty_bar + 8u * acc);   // the accumulator is free
      if (p.out && e < 4 && g < d) {   // C^T row (fp32), kept for checks of the intermediates
        float *dst = reinterpret_cast<float *>(p.out) + (size_t)bz * p.out_bstride + (size_t)g * p.out_ld;
#pragma unroll
        for (int j = 0; j < 64; j += 4)
          if (j < r) *reinterpret_cast<float4 *>(dst + j) = make_float4(cv[j], cv[j + 1], cv[j + 2], cv[j + 3]);
      }
      const int h = r / 2, i_lo = e < 4 ? 0 : h, i_hi = e < 4 ? h : r;
      if (g < d) {
        __nv_bfloat16 *op = p.cs + (size_t)bz * r * d + g;
        if (r <= 32)
          apply_rows<32>(ss.Gs, cv, i_lo, i_hi, d, op);
        else
          apply_rows<64>(ss.Gs, cv, i_lo, i_hi, d, op);
      }
      epi_bar();   // the next tile may restage ss.Gs
    }
  }
}

// Warp roles. Every issuing loop runs on one lane and is a short dependent instruction chain,
// so A and B are issued by two warps in parallel.

// PMMA: cta_group::2 pair MMAs. A kernel holding pair instructions may only be launched as a
// cluster, so the single-CTA engine is a separate instantiation without them.
template <bool PMMA>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // the next kernel of the stream may start launching now; it waits for this grid to finish
  // before it reads anything (pdl_wait), so this only overlaps launch latency and set-up
  ptx::pdl_launch_dependents();
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const uint32_t S = (uint32_t)p.stages;
  constexpr bool pmma = PMMA;
  const uint32_t a_bytes = 16384u;
  // B bytes in this CTA's shared memory per stage (half the tile for pair MMAs)
  const uint32_t b_bytes = (uint32_t)p.BN * 128u / (pmma ? 2u : 1u);
  const uint32_t stage_bytes = a_bytes + b_bytes;
  const uint32_t staging = base + p.staging_off;
  const uint32_t bar_base =
      base + p.bar_off;
  // full[S] | empty[S] | tfull[2] | tempty[2] | tmem slot
  const uint32_t full_bar = bar_base, empty_bar = bar_base + 8u * S;
  const uint32_t tfull_bar = bar_base + 16u * S, tempty_bar = tfull_bar + 16u;
  const uint32_t tmem_slot = tempty_bar + 16u;
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem + (tmem_slot - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = 128 / p.elem_bytes;   // elements in one 128-byte row
  const int crank = p.cluster == 2 ? (int)ptx::cluster_ctarank() : 0;
  const bool leader = crank == 0;
  const int cid = (int)blockIdx.x / p.cluster, ncl = (int)gridDim.x / p.cluster;
  const int mp_tiles = (p.m_tiles + p.cluster - 1) / p.cluster;
  const int total = p.batch * mp_tiles * p.n_tiles;

  if (warp == kWarpLoadA && lane == 0) {
    for (uint32_t s = 0; s < S; ++s) {
      ptx::mbar_init(full_bar + 8u * s, 2);    // the A and the B issuer
      // the MMA that reads this stage (pair MMAs: the one issuing CTA, whose commit arrives
      // on the stage barrier of both CTAs)
      ptx::mbar_init(empty_bar + 8u * s, 1u);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar + 8u * a, 1);
      // pair MMAs: the even CTA's MMA waits for the epilogues of both CTAs
      ptx::mbar_init(tempty_bar + 8u * a, (uint32_t)(kEpiWarps * (pmma ? 2 : 1)));
    }
    ptx::mbar_init_fence();
    ptx::tma_prefetch_desc(&tmA0);
    if (p.a_split < p.m_tiles) ptx::tma_prefetch_desc(&tmA1);
    if (p.tma_store) ptx::tma_prefetch_desc(&tmOut);
  }
  if (warp == kWarpLoadB && lane == 0) {
    ptx::tma_prefetch_desc(&tmB0);
    if (p.b_split < p.k_chunks) ptx::tma_prefetch_desc(&tmB1);
  }
  if (warp == kWarpMma) {
    if constexpr (PMMA) {
      ptx::tmem_alloc_pair(tmem_slot, 2u * p.acc_cols);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tmem_slot, 2u * p.acc_cols);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the peer's barriers must be initialised before its loads and commits reach them
  if (p.cluster == 2) ptx::cluster_sync_all();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;
  // set-up above overlaps the previous kernel; its outputs are read only after this
  ptx::pdl_wait();

  if (warp == kWarpLoadA) {
    // ------------------------------------------------------------ TMA producer, operand A
    if (lane == 0) {
      uint32_t s = 0, ph = 0, sa = base;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const TileCoord tc = decode_tile(t, p, mp_tiles, crank);
        // a pair's tile past the last M tile reads rows past the end of map A0 (zeros)
        const bool phantom = tc.m_tile >= p.m_tiles;
        const bool a_second = !phantom && tc.m_tile >= p.a_split;
        const int m0 = phantom ? p.a_split * 128 : (a_second ? tc.m_tile - p.a_split : tc.m_tile) * 128;
        const CUtensorMap *ma = a_second ? &tmA1 : &tmA0;
        const int a_b = (a_second ? p.a_batched1 : p.a_batched0) ? tc.bz : 0;
        const int a_k0 = p.a_kdiag > 0 ? tc.n_tile * p.a_kdiag : 0;
        const int a_k1 = p.a_k1 >= 0 ? p.a_k1 : p.b_split * chunk;
        int s_lo;
        const int kct = tile_chunks(p, tc, crank, s_lo);
        const int rc = p.k_chunks - p.b_split;
        int seg = 0, sc = 0;   // segmented mode: segment and chunk within it
        for (int kc = 0; kc < kct; ++kc) {
          if (!ptx::mbar_wait(empty_bar + 8u * s, ph ^ 1u, p.timeouts)) {
            ok = false;
            break;
          }
          const uint32_t full = full_bar + 8u * s;
          // K / row / batch coordinates and map of this chunk of A
          const CUtensorMap *mk = ma;
          int ka, arow = m0, ab = a_b;
          if (kc < p.b_split) {
            ka = a_k0 + kc * chunk;
          } else if (p.seg_n > 0) {
            const int sg = s_lo + seg;
            mk = &tmA1;
            ka = a_k1 + sc * chunk;
            arow = tc.m_tile * 128 - sg * p.seg_n;
            ab = sg;
            if (++sc == rc) {
              sc = 0;
              ++seg;
            }
          } else {
            ka = a_k1 + (kc - p.b_split) * chunk;
          }
          if constexpr (PMMA) {
            // both CTAs' A land on the even CTA's full barrier, which expects them all
            if (leader) ptx::mbar_arrive_expect_tx(full, 2u * a_bytes);
            ptx::tma_load_3d_pair(sa, mk, ptx::mapa_shared(full, 0), ka, arow, ab);
          } else if (p.a_major == 0) {
            ptx::mbar_arrive_expect_tx(full, a_bytes);
            ptx::tma_load_3d(sa, mk, full, ka, arow, ab);
          } else {
            ptx::mbar_arrive_expect_tx(full, a_bytes);
            for (int i = 0; i < 128 / chunk; ++i)
              ptx::tma_load_3d(sa + (uint32_t)(i * chunk * 128), ma, full, m0 + i * chunk,
                               kc * chunk, a_b);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
            sa = base;
          } else {
            sa += stage_bytes;
          }
        }
      }
    }
  } else if (warp == kWarpLoadB) {
    // ------------------------------------------------------------ TMA producer, operand B
    if (lane == 0) {
      uint32_t s = 0, ph = 0, sb = base + a_bytes;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const TileCoord tc = decode_tile(t, p, mp_tiles, crank);
        const int n0 = tc.n_tile * p.BN;
        const int b_b0 = p.b_batched0 ? tc.bz : 0, b_b1 = p.b_batched1 ? tc.bz : 0;
        int s_lo;
        const int kct = tile_chunks(p, tc, crank, s_lo);
        const int rc = p.k_chunks - p.b_split;
        int seg = 0, sc = 0;
        for (int kc = 0; kc < kct; ++kc) {
          if (!ptx::mbar_wait(empty_bar + 8u * s, ph ^ 1u, p.timeouts)) {
            ok = false;
            break;
          }
          const uint32_t full = full_bar + 8u * s;
          const bool b_second = kc >= p.b_split;
          const CUtensorMap *mb = b_second ? &tmB1 : &tmB0;
          int kk = b_second ? kc - p.b_split : kc;
          int b_b = b_second ? b_b1 : b_b0;
          if (b_second && p.seg_n > 0) {
            kk = sc;
            b_b = s_lo + seg;
            if (++sc == rc) {
              sc = 0;
              ++seg;
            }
          }
          if constexpr (PMMA) {
            if (leader) ptx::mbar_arrive_expect_tx(full, 2u * b_bytes);
            const uint32_t fb = ptx::mapa_shared(full, 0);
            const int half = p.BN / 2;
            if ((b_second ? p.b_major1 : p.b_major) == 0) {
              ptx::tma_load_3d_pair(sb, mb, fb, kk * chunk, n0 + crank * half, b_b);
            } else {
              for (int i = 0; i < half / chunk; ++i)
                ptx::tma_load_3d_pair(sb + (uint32_t)(i * chunk * 128), mb, fb,
                                      n0 + crank * half + i * chunk, kk * chunk, b_b);
            }
          } else {
            ptx::mbar_arrive_expect_tx(full, b_bytes);
            if ((b_second ? p.b_major1 : p.b_major) == 0) {
              ptx::tma_load_3d(sb, mb, full, kk * chunk, n0, b_b);
            } else {
              for (int i = 0; i < p.BN / chunk; ++i)
                ptx::tma_load_3d(sb + (uint32_t)(i * chunk * 128), mb, full, n0 + i * chunk,
                                 kk * chunk, b_b);
            }
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
            sb = base + a_bytes;
          } else {
            sb += stage_bytes;
          }
        }
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issue
    // (pair MMAs: only the even CTA issues, for both CTAs of the pair)
    if (lane == 0 && (!pmma || leader)) {
      // K-major SW128: rows of 128 B, 8-row groups 1024 B apart (SBO), K advance inside the row.
      // MN-major SW128: 128-byte rows hold `chunk` MN elements; MN groups LBO apart, 8-row K
      // groups 1024 B apart; one MMA consumes 32 bytes of K = 32/elem rows.
      const uint32_t mn_lbo = (uint32_t)(chunk * 128);
      const uint32_t mn_kstep16 = (4096u / (uint32_t)p.elem_bytes) >> 4;
      const uint64_t a_desc0 = ptx::sdesc_sw128(base, p.a_major ? mn_lbo : 16u, 1024u);
      const uint64_t b_desc0 = ptx::sdesc_sw128(base + a_bytes, p.b_major ? mn_lbo : 16u, 1024u);
      const uint64_t b_desc1 = ptx::sdesc_sw128(base + a_bytes, p.b_major1 ? mn_lbo : 16u, 1024u);
      const uint32_t a_k16 = p.a_major ? mn_kstep16 : 2u;
      const uint32_t b_k16_0 = p.b_major ? mn_kstep16 : 2u;
      const uint32_t b_k16_1 = p.b_major1 ? mn_kstep16 : 2u;
      const uint32_t st16 = stage_bytes >> 4;
      const bool f16 = p.elem_bytes == 2;
      uint32_t s = 0, ph = 0, soff = 0, i = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl, ++i) {
        const uint32_t acc = i & 1u;
        if (!ptx::mbar_wait(tempty_bar + 8u * acc, ((i >> 1) & 1u) ^ 1u, p.timeouts)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * p.acc_cols;
        int s_lo;
        const int kct = p.seg_n > 0 ? tile_chunks(p, decode_tile(t, p, mp_tiles, crank), crank, s_lo)
                                    : p.k_chunks;
        for (int kc = 0; kc < kct; ++kc) {
          if (!ptx::mbar_wait(full_bar + 8u * s, ph, p.timeouts)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const bool b_second = kc >= p.b_split;
          const uint64_t ad = a_desc0 + soff;
          const uint64_t bd = (b_second ? b_desc1 : b_desc0) + soff;
          const uint32_t bk = b_second ? b_k16_1 : b_k16_0;
          const uint32_t idesc = b_second ? p.idesc1 : p.idesc;
          if constexpr (PMMA) {
            if (f16) {
#pragma unroll
              for (uint32_t ks = 0; ks < 4; ++ks)
                ptx::tc_mma_f16_pair(d_tmem, ad + ks * a_k16, bd + ks * bk, idesc, (kc | ks) ? 1u : 0u);
            } else {
#pragma unroll
              for (uint32_t ks = 0; ks < 4; ++ks)
                ptx::tc_mma_tf32_pair(d_tmem, ad + ks * a_k16, bd + ks * bk, idesc, (kc | ks) ? 1u : 0u);
            }
            // frees the stage in both CTAs when these MMAs finish
            ptx::tc_commit_pair_mc(empty_bar + 8u * s, (uint16_t)3);
          } else {
            if (f16) {
#pragma unroll
              for (uint32_t ks = 0; ks < 4; ++ks)
                ptx::tc_mma_f16(d_tmem, ad + ks * a_k16, bd + ks * bk, idesc, (kc | ks) ? 1u : 0u);
            } else {
#pragma unroll
              for (uint32_t ks = 0; ks < 4; ++ks)
                ptx::tc_mma_tf32(d_tmem, ad + ks * a_k16, bd + ks * bk, idesc, (kc | ks) ? 1u : 0u);
            }
            // frees the smem stage when these MMAs finish
            ptx::tc_commit(empty_bar + 8u * s);
          }
          if (++s == S) {
            s = 0;
            ph ^= 1u;
            soff = 0;
          } else {
            soff += st16;
          }
        }
        if (ok) {   // accumulator ready (in both CTAs of a pair)
          if constexpr (PMMA)
            ptx::tc_commit_pair_mc(tfull_bar + 8u * acc, (uint16_t)3);
          else
            ptx::tc_commit(tfull_bar + 8u * acc);
        }
      }
    }
  } else if (warp >= kEpiWarp0) {
    // ------------------------------------------------------------ epilogue
    const int e = warp - kEpiWarp0;
    const int q = warp & 3;   // TMEM lane quarter this warp may read
    // column split of a tile between the two warps of a quarter, in 32-column units
    const int units = p.BN / 32 + ((p.BN % 32) ? 1 : 0);
    const int u_lo = (e < 4) ? 0 : (units + 1) / 2;
    const int u_hi = (e < 4) ? (units + 1) / 2 : units;
    const int c_lo = u_lo * 32, c_hi = u_hi * 32 < p.BN ? u_hi * 32 : p.BN;
    // this warp's staging tiles: epi_bufs pairs, used in turn
    const uint32_t stg = staging + (uint32_t)e * (uint32_t)p.epi_bufs * kStagingPairBytes;
    const bool add_bias = p.tma_store && p.bias;
    uint32_t buf_i = 0, i = 0;
    TileCoord tcn = decode_tile(cid < total ? cid : 0, p, mp_tiles, crank);
    if (p.epi == EPI_CG_SOLVE) {
      cg_solve_epilogue(p, smem, base, tmem_base, tfull_bar, tempty_bar, cid, ncl, total,
                        mp_tiles, e, lane, c_lo, c_hi);
    }
    for (int t = p.epi == EPI_CG_SOLVE ? total : cid; t < total; t += ncl, ++i) {
      const uint32_t acc = i & 1u;
      const TileCoord tc = tcn;
      if (t + ncl < total) tcn = decode_tile(t + ncl, p, mp_tiles, crank);
      int got = 0;
      if (lane == 0) got = ptx::mbar_wait(tfull_bar + 8u * acc, (i >> 1) & 1u, p.timeouts) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      ptx::tc_fence_after();
      if (tc.m_tile >= p.m_tiles) {   // a pair's tile past the last M tile: nothing to store
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (pmma && !leader)
            ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar + 8u * acc, 0));
          else
            ptx::mbar_arrive(tempty_bar + 8u * acc);
        }
        continue;
      }
      const bool second = tc.m_tile >= p.a_split;
      const int m0 = (second ? tc.m_tile - p.a_split : tc.m_tile) * 128;
      const int n0 = tc.n_tile * p.BN;
      const uint32_t taddr = tmem_base + acc * p.acc_cols + ((uint32_t)(q * 32) << 16);
      const int cols_lim = second ? p.cols2_valid : p.cols_valid;
      if (p.tma_store) {
        // bf16 rows. A warp has at most 128 columns of a tile: up to four 32-column pieces,
        // handled in pairs. Both TMEM loads of a pair complete (tcgen05.wait::ld) before any
        // other instruction touches their registers -- the destination registers of an
        // outstanding tcgen05.ld are not yet written, and the compiler does not know that.
        // Each piece then gets the staged bias and is packed to bf16 into a 64B-swizzled
        // 32 x 32 staging tile; a pair goes out as one bulk group of TMA stores. The warp
        // alternates two pairs of staging tiles and reuses a pair only after the group that
        // last read it has finished reading.
        const int row0 = m0 + q * 32;
        int npc = 0;   // pieces inside the tile's and the tensor's columns (uniform)
#pragma unroll
        for (int s = 0; s < 4; ++s)
          if (c_lo + 32 * s < c_hi && n0 + c_lo + 32 * s < cols_lim) npc = s + 1;
        if (row0 < p.rows_valid) {   // else the 32-row slab is outside the tensor
          const int zb = p.out_batched ? tc.bz : 0;
#pragma unroll
          for (int s0 = 0; s0 < 4; s0 += 2) {
            if (s0 < npc) {
              const bool two = s0 + 1 < npc;
              uint32_t v[2][32];
              ptx::tmem_ld32(taddr + (uint32_t)(c_lo + 32 * s0), v[0]);
              if (two) ptx::tmem_ld32(taddr + (uint32_t)(c_lo + 32 * s0 + 32), v[1]);
              ptx::tmem_ld_wait();
              if (add_bias) {   // every lane reads the same bytes: one broadcast line per load
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  // the bias array is padded to a multiple of 256 columns (no bound check)
                  const float4 *b4 =
                      reinterpret_cast<const float4 *>(p.bias + n0 + c_lo + 32 * (s0 + h));
#pragma unroll
                  for (int j = 0; j < 8; ++j) {
                    const float4 bb = __ldg(b4 + j);
                    v[h][4 * j + 0] = __float_as_uint(__uint_as_float(v[h][4 * j + 0]) + bb.x);
                    v[h][4 * j + 1] = __float_as_uint(__uint_as_float(v[h][4 * j + 1]) + bb.y);
                    v[h][4 * j + 2] = __float_as_uint(__uint_as_float(v[h][4 * j + 2]) + bb.z);
                    v[h][4 * j + 3] = __float_as_uint(__uint_as_float(v[h][4 * j + 3]) + bb.w);
                  }
                }
              }
              if (p.act == 1) {
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    v[h][j] = __float_as_uint(gelu_erf(__uint_as_float(v[h][j])));
              }
              // the pair about to be overwritten has been read by the group that stored it
              if (lane == 0) {
                if (p.epi_bufs > 1)
                  ptx::bulk_wait_read<1>();
                else
                  ptx::bulk_wait_read<0>();
              }
              __syncwarp();
              const uint32_t buf = stg + buf_i * kStagingPairBytes;
              stage_bits32(buf, lane, v[0]);
              if (two) stage_bits32(buf + 2048u, lane, v[1]);
              ptx::fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                ptx::tma_store_3d(&tmOut, buf, n0 + c_lo + 32 * s0, row0, zb);
                if (two) ptx::tma_store_3d(&tmOut, buf + 2048u, n0 + c_lo + 32 * s0 + 32, row0, zb);
                ptx::bulk_commit();
              }
              if (++buf_i == (uint32_t)p.epi_bufs) buf_i = 0;
            }
          }
        }
      } else {
        const long long g = (long long)m0 + q * 32 + lane;
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
          const int col0 = n0 + c0;
          if (col0 >= cols_lim) break;   // uniform across the warp
          if (c0 + 32 <= p.BN) {
            uint32_t v[32];
            ptx::tmem_ld32(taddr + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            float f[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = __uint_as_float(v[j]);
            epilogue16(p, f, g, col0, tc.bz, second);
            epilogue16(p, f + 16, g, col0 + 16, tc.bz, second);
          } else {
            uint32_t v[16];
            ptx::tmem_ld16(taddr + (uint32_t)c0, v);
            ptx::tmem_ld_wait();
            float f[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(v[j]);
            epilogue16(p, f, g, col0, tc.bz, second);
          }
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {   // this accumulator may be overwritten (pair MMAs: by the even CTA)
        if (pmma && !leader)
          ptx::mbar_arrive_cluster(ptx::mapa_shared(tempty_bar + 8u * acc, 0));
        else
          ptx::mbar_arrive(tempty_bar + 8u * acc);
      }
    }
    if (p.tma_store && lane == 0) ptx::bulk_wait<0>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA of a pair leaves while the other may still write its shared memory or
  // arrive on its barriers
  if (p.cluster == 2) ptx::cluster_sync_all();
  if (warp == kWarpMma) {
    ptx::tc_fence_after();
    if constexpr (PMMA)
      ptx::tmem_dealloc_pair(tmem_base, 2u * p.acc_cols);
    else
      ptx::tmem_dealloc(tmem_base, 2u * p.acc_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

bool encode(CUtensorMap *map, const TcOperand &op, cuuint32_t box0, cuuint32_t box1,
            CUtensorMapSwizzle sw) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return false;
  const CUtensorMapDataType dt =
      op.elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  long long bstride = op.batch_stride;
  if (op.batch <= 1) bstride = ((op.rows * op.row_stride) + 15) / 16 * 16;
  cuuint64_t dims[3] = {(cuuint64_t)op.inner, (cuuint64_t)op.rows,
                        (cuuint64_t)(op.batch < 1 ? 1 : op.batch)};
  cuuint64_t strides[2] = {(cuuint64_t)op.row_stride, (cuuint64_t)bstride};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, dt, 3, const_cast<void *>(op.base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, []() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 148;
  });
  return n;
}

}  // namespace

uint32_t tc_idesc(int elem_bytes, int a_major, int b_major, int n, int m) {
  const uint32_t fmt = elem_bytes == 2 ? 1u : 2u;   // BF16 = 1, TF32 = 2
  uint32_t d = 0;
  d |= 1u << 4;                          // D format: F32
  d |= fmt << 7;                         // A format
  d |= fmt << 10;                        // B format
  d |= (uint32_t)(a_major & 1) << 15;    // A major (1 = MN)
  d |= (uint32_t)(b_major & 1) << 16;    // B major
  d |= ((uint32_t)n >> 3) << 17;         // N / 8
  d |= ((uint32_t)m >> 4) << 24;         // M / 16
  return d;
}

bool tc_make_map(CUtensorMap *map, const TcOperand &op, int box_rows) {
  return encode(map, op, (cuuint32_t)(128 / op.elem_bytes), (cuuint32_t)box_rows,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tc_make_store_map(CUtensorMap *map, const TcOperand &op) {
  return encode(map, op, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

// Co-resident 2-CTA clusters for this kernel and shared-memory size (a persistent grid larger
// than that would run a second, mostly idle wave). Queried once per (kernel, size) and cached;
// a failed query is cleared and falls back to one pair per two SMs.
static int max_active_pairs(void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                                         CUtensorMap, TcGemmParams),
                            cudaLaunchConfig_t cfg, bool pmma) {
  static std::mutex mu;
  static std::map<std::pair<int, uint64_t>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_pair(dev, ((uint64_t)cfg.dynamicSmemBytes << 1) | (pmma ? 1u : 0u));
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  // the query takes the cluster shape alone
  cudaLaunchAttribute cl = {};
  cl.id = cudaLaunchAttributeClusterDimension;
  cl.val.clusterDim.x = 2;
  cl.val.clusterDim.y = 1;
  cl.val.clusterDim.z = 1;
  cfg.attrs = &cl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(2, 1, 1);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = num_sms() / 2;
  }
  cache[key] = n;
  return n;
}

cudaError_t tc_gemm_launch(TcGemmParams p, const CUtensorMap &a0, const CUtensorMap &a1,
                           const CUtensorMap &b0, const CUtensorMap &b1,
                           const CUtensorMap &out_map, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(tc_gemm_kernel<false>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(tc_gemm_kernel<true>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
  });
  if (attr_err != cudaSuccess) return attr_err;
  if (p.m_tiles <= 0 || p.n_tiles <= 0 || p.batch <= 0 || p.k_chunks <= 0) return cudaSuccess;
  // MN-major tf32 operands need the 32-byte-atom 128B swizzle, which this engine does not
  // set up; every tf32 use here is K-major.
  if (p.elem_bytes == 4 && (p.a_major || p.b_major || p.b_major1)) return cudaErrorNotSupported;
  if (p.BN < 16 || p.BN > 256 || p.BN % 16) return cudaErrorInvalidValue;
  if (p.tma_store && (p.epi != EPI_ROW_BF16 || p.BN % 32)) return cudaErrorInvalidValue;
  if ((p.b_major || p.b_major1) && p.BN % 64) return cudaErrorInvalidValue;
  p.acc_cols = 32;
  while (p.acc_cols < (uint32_t)p.BN) p.acc_cols <<= 1;
  if (p.seg_n > 0 && (p.batch != 1 || p.a_major || p.seg_count <= 0 || p.k_chunks <= p.b_split))
    return cudaErrorInvalidValue;
  p.cluster = 1;
  if (p.pair_mma) {
    p.cluster = 2;
    if (p.BN % 32) return cudaErrorInvalidValue;                   // halves of whole 8-row groups
    if ((p.b_major || p.b_major1) && p.BN % 128) return cudaErrorInvalidValue;
    if (p.a_major) return cudaErrorNotSupported;
  }
  const uint32_t stage = 16384u + (uint32_t)p.BN * 128u / (p.pair_mma ? 2u : 1u);
  // Epilogue staging: two pairs of tiles per warp when a tile's main loop is short (the
  // epilogue then sets the pace and alternates pairs without waiting), one pair otherwise,
  // which leaves room for more pipeline stages to hide the operand loads' latency.
  if (p.epi_bufs != 1 && p.epi_bufs != 2) p.epi_bufs = p.k_chunks <= 6 ? 2 : 1;
  uint32_t staging = p.tma_store ? (uint32_t)kEpiWarps * (uint32_t)p.epi_bufs * kStagingPairBytes : 0u;
  if (p.epi == EPI_CG_SOLVE) {
    if (p.pair_mma || p.n_tiles != 1 || p.m_tiles != p.a_split + 1 || !p.g_first ||
        p.solve_r <= 0 || p.solve_r > 64 || p.solve_r % 4 || p.BN < p.solve_r)
      return cudaErrorInvalidValue;
    staging = ((uint32_t)sizeof(SolveSmem) + 1023u) & ~1023u;
  }
  const uint32_t fixed = 1024u + staging + 256u;   // alignment slack, staging, barriers
  int S = (int)((232448u - fixed) / stage);
  if (S > 8) S = 8;
  if (S < 2) return cudaErrorInvalidValue;
  p.stages = S;
  p.staging_off = (uint32_t)S * stage;
  p.solve_off = p.staging_off;
  p.bar_off = p.staging_off + staging;   // barriers follow the staging buffers
  uint32_t smem = (uint32_t)S * stage + fixed;
  // one CTA per SM: the two accumulators may take all 512 TMEM columns
  if (smem < 116u * 1024u) smem = 116u * 1024u;
  p.smem_bytes = smem;
  const long long units =
      (long long)p.batch * ((p.m_tiles + p.cluster - 1) / p.cluster) * p.n_tiles;
  // programmatic stream serialization: this grid may launch while the previous kernel of
  // the stream finishes (the kernel waits for it with pdl_wait before reading)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.cluster == 1) {
    cfg.gridDim = dim3((unsigned)(units < num_sms() ? units : num_sms()), 1, 1);
    return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<false>, a0, a1, b0, b1, out_map, p);
  }
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.numAttrs = 2;
  auto kern = tc_gemm_kernel<true>;
  const int max_clusters = max_active_pairs(kern, cfg, true);
  const long long clusters = units < max_clusters ? units : max_clusters;
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, a0, a1, b0, b1, out_map, p);
}

}  // namespace dyra
