// Newton-Schulz inverse of the per-sample Gram matrix for larger r ("DyRA" summary page, 2.4:
// Newton-Schulz for larger r, on tensor cores): the start, every iteration and the finish in
// one kernel.
//
// Start (Jacobi scaling): D = diag(G + lambda I)^-1/2, G_hat = D (G + lambda I) D,
// alpha = 1 / max_i sum_j |G_hat_ij|, X0 = alpha I, E0 = I - alpha G_hat. One iteration of
// X <- X (2I - G_hat X) is, with E = I - G_hat X (E and X are polynomials in G_hat, hence
// symmetric and commuting),
//     X' = X (2I - G_hat X) = X + X E,        E' = I - G_hat X' = E E,
// two products per iteration (the last iteration forms X' only). X = Z + alpha I where Z
// starts at 0 and collects the products X E: Z stays in the tensor memory accumulator of its
// tile across iterations (fp32), the identity part is never rounded, and the iterate written
// for the other tiles is Z + alpha I. The kernel finishes with G^-1 = D X_T D.
//
// A cluster of 2 rt^2 CTAs (rt = ceil(r / 128)) takes one sample: CTA c owns the 128 x 128
// output tile (row block c / rt of [E ; X], column block c % rt). At the start each CTA reads
// the whole diagonal of G, the row sums of |G_hat| for every nc-th row (the maximum goes to
// the cluster through distributed shared memory, in a fixed order) and writes its own tile of
// E0 or X0. Per iteration it streams the K chunks of its A rows (E or X) and of its B operand
// (rows of E: E is symmetric, so B^T = B) by TMA from the iterate in global memory
// (L2-resident) into a ring of shared-memory stages and accumulates the tf32 products in TMEM
// (tcgen05.mma, issued by one thread). The epilogue warps stage the tile, 32 columns at a
// time, in the idle ring buffers (128-byte swizzle) and write it with TMA stores. The iterates
// alternate between two buffers. Between iterations the stores complete and every thread of
// the cluster meets at a cluster barrier (release / acquire), so the next iteration's loads
// see the whole new iterate; every thread executes every barrier, whatever its role did, so a
// wait that gives up cannot leave a peer blocked.
//
// Warps: 0 TMA producer (one lane), 1 TMEM allocation and MMA issue (one lane), 4..7 epilogue
// (warp w reads TMEM lane quarter w % 4, i.e. rows 32 (w % 4) .. + 31 of the tile); all eight
// take part in the start.
#include "kernels.cuh"
#include "ptx.cuh"
#include "tc_gemm.cuh"

#include <cuda_bf16.h>
#include <mutex>

namespace dyra {

namespace {

constexpr int kNsfThreads = 256;
constexpr int kNsfStages = 6;
constexpr uint32_t kNsfStageBytes = 2 * 16384;   // A and B chunks: 128 rows x 128 bytes each
constexpr uint32_t kNsfSmem = 1024 + kNsfStages * kNsfStageBytes + 256;
constexpr int kEpiBarrier = 1;                    // named barrier of the 4 epilogue warps
constexpr int kNsMaxR = 256;

struct NsParams {
  int r, rt, iters;
  float ridge;
  const float *G;              // [batch][r][r] fp32 (without the ridge)
  float *ex0, *ex1;            // iterate buffers, [batch][2r][r] fp32 each ([E ; X])
  float *G32;                  // [batch][r][r] fp32 G^-1
  __nv_bfloat16 *Ginv;         // [batch][r][r] bf16 G^-1
  int *status;                 // [0] samples set to 0, [1] bounded waits that gave up
  uint32_t idesc;
};

// The four tensor maps of the two iterate buffers: E and X blocks of each ([batch][r][r],
// box {32, 128}, 128-byte swizzle), used for the TMA loads and for the TMA stores.
struct NsMaps {
  CUtensorMap m[2][2];
};

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ int ld_cluster_s32(const int *p, uint32_t rank) {
  int v;
  asm volatile("ld.shared::cluster.b32 %0, [%1];"
               : "=r"(v)
               : "r"(ptx::mapa_shared(ptx::smem_u32(p), rank))
               : "memory");
  return v;
}

__device__ __forceinline__ float ld_cluster_f32(const float *p, uint32_t rank) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];"
               : "=f"(v)
               : "r"(ptx::mapa_shared(ptx::smem_u32(p), rank))
               : "memory");
  return v;
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync %0, 128;" ::"n"(kEpiBarrier) : "memory");
}

// 32 fp32 values of row `row` (0..127) into a 128 x 32 staging tile with the 128-byte
// swizzle TMA uses (16-byte chunk c of row i at chunk c ^ (i % 8)); `diag` >= 0 adds `add`
// to column diag of the row.
__device__ __forceinline__ void stage_row32(uint32_t buf, int row, const uint32_t *v, int diag,
                                            float add) {
  const uint32_t dst = buf + (uint32_t)row * 128u;
  const uint32_t sw = (uint32_t)(row & 7);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      w[k] = __uint_as_float(v[4 * c + k]) + ((4 * c + k) == diag ? add : 0.f);
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(dst + (((uint32_t)c ^ sw) << 4)),
                 "f"(w[0]), "f"(w[1]), "f"(w[2]), "f"(w[3])
                 : "memory");
  }
}

__global__ void __launch_bounds__(kNsfThreads, 1)
    ns_fused_kernel(const __grid_constant__ NsMaps maps, const __grid_constant__ NsParams p) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float sd[kNsMaxR];   // D
  __shared__ float red[kNsfThreads / 32];
  __shared__ float cmax, alpha_s;
  __shared__ int bad_cta;
  __shared__ int bad_all;
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  const uint32_t bar_base = base + kNsfStages * kNsfStageBytes;
  const uint32_t full_bar = bar_base, empty_bar = bar_base + 8u * kNsfStages;
  const uint32_t tfull_bar = bar_base + 16u * kNsfStages;
  const uint32_t tmem_slot = tfull_bar + 8u;
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem_raw + (tmem_slot - raw_addr));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = (int)ptx::cluster_ctarank(), nc = (int)ptx::cluster_nctarank();
  const int b = blockIdx.y;
  const int r = p.r, rt = p.rt;
  const int rb = c / rt, cb = c % rt;            // row block of [E ; X], column block
  const bool x_tile = rb >= rt;                  // this CTA's rows are rows of X
  const int row0 = (x_tile ? rb - rt : rb) * 128;  // first row inside E or X
  const int col0 = cb * 128;
  const int kchunks = (r + 31) / 32;             // 32 fp32 of K per 128-byte chunk
  int *timeouts = p.status + 1;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < kNsfStages; ++s) {
      ptx::mbar_init(full_bar + 8u * s, 1);
      ptx::mbar_init(empty_bar + 8u * s, 1);
    }
    ptx::mbar_init(tfull_bar, 1);
    ptx::mbar_init_fence();
    for (int i = 0; i < 2; ++i)
      for (int j = 0; j < 2; ++j) ptx::tma_prefetch_desc(&maps.m[i][j]);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 128);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot_ptr;
  // the apply GEMM may start launching now (it waits for this grid to finish before reading)
  ptx::pdl_launch_dependents();
  // G comes from the previous kernel of the stream: nothing is read before this wait
  ptx::pdl_wait();

  // ------------------------------------------------------------ start
  // D from the whole diagonal (every CTA reads it: the flag of a diagonal entry that is not
  // positive and finite is the same in every CTA of the sample)
  const float *g = p.G + (size_t)b * r * r;
  bool bad = false;
  if (tid < r) {
    const float gii = __ldcg(g + (size_t)tid * r + tid) + p.ridge;
    bad = !(gii > 0.f && gii < INFINITY);
    sd[tid] = bad ? 0.f : rsqrtf(gii);
  }
  bad = __syncthreads_or(bad) != 0;
  // row sums of |G_hat| of rows c, c + nc, ... (warp w takes every 8th of them)
  float rmax = 0.f;
  for (int i = c + nc * warp; i < r; i += nc * (kNsfThreads / 32)) {
    const float *gr = g + (size_t)i * r;
    float s = 0.f;
    for (int j = lane; j < r; j += 32)
      s += fabsf((__ldcg(gr + j) + (i == j ? p.ridge : 0.f)) * sd[i] * sd[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    rmax = fmaxf(rmax, s);
  }
  if (lane == 0) red[warp] = rmax;
  __syncthreads();
  if (tid == 0) {
    float m = 0.f;
    for (int k = 0; k < kNsfThreads / 32; ++k) m = fmaxf(m, red[k]);
    cmax = m;
  }
  ptx::cluster_sync_all();   // every CTA's cmax is written
  if (tid == 0) {
    float m = 0.f;
    for (int k = 0; k < nc; ++k) m = fmaxf(m, ld_cluster_f32(&cmax, (uint32_t)k));
    // a flagged sample starts from E0 = I, X0 = 0: every iterate and its G^-1 stay 0
    alpha_s = (bad || !(m > 0.f)) ? 0.f : 1.f / m;
  }
  __syncthreads();
  const float alpha = alpha_s;
  {
    // this CTA's tile of the start: E0 = I - alpha G_hat (E tiles) or X0 = alpha I (X tiles)
    float *dst = (x_tile ? p.ex0 + (size_t)r * r : p.ex0) + (size_t)b * 2 * r * r;
    for (int e = tid; e < 128 * 32; e += kNsfThreads) {
      const int i = row0 + e / 32, j = col0 + 4 * (e % 32);
      if (i < r && j < r) {   // r % 8 == 0: a group of 4 columns is inside or outside
        float v[4];
        if (x_tile) {
#pragma unroll
          for (int k = 0; k < 4; ++k) v[k] = i == j + k ? alpha : 0.f;
        } else {
          const float4 gv = __ldcg(reinterpret_cast<const float4 *>(g + (size_t)i * r + j));
          const float gg[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float gh = (gg[k] + (i == j + k ? p.ridge : 0.f)) * sd[i] * sd[j + k];
            v[k] = (i == j + k ? 1.f : 0.f) - alpha * gh;
          }
        }
        *reinterpret_cast<float4 *>(dst + (size_t)i * r + j) = make_float4(v[0], v[1], v[2], v[3]);
      }
    }
  }
  // the start is in global memory, visible to the TMA loads of every CTA of the cluster
  fence_proxy_async_global();
  ptx::cluster_sync_all();
  fence_proxy_async_global();

  bool ok = true;                    // this thread's bounded waits all completed
  uint32_t ring = 0, ring_ph = 0;    // producer / MMA position in the stage ring
  const int q = warp & 3;
  const uint32_t taddr = tmem + ((uint32_t)(32 * q) << 16);
  for (int t = 0; t < p.iters; ++t) {
    const bool last = t + 1 == p.iters;
    const bool active = !(last && !x_tile);      // the last iteration forms X' only
    const int src = t & 1;
    const CUtensorMap *mA = &maps.m[src][x_tile ? 1 : 0];
    const CUtensorMap *mB = &maps.m[src][0];
    if (active && warp == 0 && lane == 0) {
      // ------------------------------------------------------------ TMA producer
      uint32_t s = ring, ph = ring_ph;
      for (int kc = 0; kc < kchunks; ++kc) {
        if (ok && !ptx::mbar_wait(empty_bar + 8u * s, ph ^ 1u, timeouts)) ok = false;
        if (ok) {
          const uint32_t sa = base + s * kNsfStageBytes;
          ptx::mbar_arrive_expect_tx(full_bar + 8u * s, kNsfStageBytes);
          ptx::tma_load_3d(sa, mA, full_bar + 8u * s, kc * 32, row0, b);
          ptx::tma_load_3d(sa + 16384u, mB, full_bar + 8u * s, kc * 32, col0, b);
        }
        if (++s == kNsfStages) {
          s = 0;
          ph ^= 1u;
        }
      }
    } else if (active && warp == 1 && lane == 0) {
      // ------------------------------------------------------------ MMA issue
      // E' = E E starts from 0; Z' = Z + X E accumulates onto Z (0 before the first iteration)
      const uint32_t keep = (x_tile && t > 0) ? 1u : 0u;
      uint32_t s = ring, ph = ring_ph;
      const uint64_t a0 = ptx::sdesc_sw128(base, 16u, 1024u);
      const uint64_t b0 = ptx::sdesc_sw128(base + 16384u, 16u, 1024u);
      const uint32_t st16 = kNsfStageBytes >> 4;
      for (int kc = 0; kc < kchunks; ++kc) {
        if (ok && !ptx::mbar_wait(full_bar + 8u * s, ph, timeouts)) ok = false;
        if (ok) {
          ptx::tc_fence_after();
          const uint64_t soff = (uint64_t)(s * st16);
#pragma unroll
          for (uint32_t ks = 0; ks < 4; ++ks)   // 4 MMAs of K = 8 (32 bytes) per chunk
            ptx::tc_mma_tf32(tmem, a0 + soff + 2 * ks, b0 + soff + 2 * ks, p.idesc,
                             (kc | ks) ? 1u : keep);
          ptx::tc_commit(empty_bar + 8u * s);
        }
        if (++s == kNsfStages) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (ok) ptx::tc_commit(tfull_bar);
    } else if (active && warp >= 4) {
      // ------------------------------------------------------------ epilogue
      int got = 0;
      if (lane == 0 && ok) got = ptx::mbar_wait(tfull_bar, (uint32_t)(t & 1), timeouts) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) ok = false;
      ptx::tc_fence_after();
      if (!last) {
        // every ring stage has been consumed by this iteration's MMAs: the ring holds the
        // staging tiles (piece pc at stage pc); X tiles write Z' + alpha I
        const int row = 32 * q + lane;
        const int dst = src ^ 1;
        for (int pc = 0; pc < 4; ++pc) {
          const int j0 = col0 + 32 * pc;
          if (j0 >= r) break;                   // uniform across the CTA
          uint32_t v[32];
          ptx::tmem_ld32(taddr + (uint32_t)(32 * pc), v);
          ptx::tmem_ld_wait();
          const uint32_t buf = base + (uint32_t)pc * kNsfStageBytes;
          const int dcol = row0 + row - j0;
          stage_row32(buf, row, v, (x_tile && dcol >= 0 && dcol < 32) ? dcol : -1, alpha);
          ptx::fence_proxy_async_smem();
          epi_sync();
          if (warp == 4 && lane == 0 && got) {
            ptx::tma_store_3d(&maps.m[dst][x_tile ? 1 : 0], buf, j0, row0, b);
            ptx::bulk_commit();
          }
        }
        // the new iterate is in global memory before the barrier releases the cluster
        if (warp == 4 && lane == 0) ptx::bulk_wait<0>();
        epi_sync();
      }
      ptx::tc_fence_before();
    }
    if (!last) {
      fence_proxy_async_global();
      ptx::cluster_sync_all();
      fence_proxy_async_global();
    }
    // the ring position after this iteration's chunks (same in every role)
    if (active) {
      for (int kc = 0; kc < kchunks; ++kc)
        if (++ring == kNsfStages) {
          ring = 0;
          ring_ph ^= 1u;
        }
    }
  }

  // ------------------------------------------------------------ finish: G^-1 = D X_T D
  // The X tiles' accumulators hold Z_T = X_T - alpha I. A sample whose start was flagged, or
  // whose result is not finite anywhere, gets G^-1 = 0 and is counted once.
  if (threadIdx.x == 0) bad_cta = 0;
  __syncthreads();
  const int i = row0 + 32 * q + lane;
  bool nonfinite = false;
  if (x_tile && warp >= 4) {
    for (int pc = 0; pc < 4; ++pc) {
      const int j0 = col0 + 32 * pc;
      if (j0 >= r) break;
      uint32_t v[32];
      ptx::tmem_ld32(taddr + (uint32_t)(32 * pc), v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (i < r && j0 + j < r) nonfinite = nonfinite || !(fabsf(__uint_as_float(v[j])) < INFINITY);
    }
    if (!ok) nonfinite = true;
  }
  if (nonfinite) bad_cta = 1;
  // the cluster agrees on the sample's flag before anything is written
  ptx::cluster_sync_all();
  if (threadIdx.x == 0) {
    int any = bad ? 1 : 0;
    for (int k = 0; k < nc; ++k) any |= ld_cluster_s32(&bad_cta, (uint32_t)k);
    bad_all = any;
    if (any && c == 0) atomicAdd(p.status, 1);
  }
  ptx::cluster_sync_all();   // no CTA leaves while a peer may still read its flag
  if (x_tile && warp >= 4) {
    const bool zero = bad_all != 0;
    const float di = i < r ? sd[i] : 0.f;
    for (int pc = 0; pc < 4; ++pc) {
      const int j0 = col0 + 32 * pc;
      if (j0 >= r) break;
      uint32_t v[32];
      ptx::tmem_ld32(taddr + (uint32_t)(32 * pc), v);
      ptx::tmem_ld_wait();
      if (i < r) {
        const size_t o = (size_t)b * r * r + (size_t)i * r + j0;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          if (j0 + j >= r) break;   // r % 8 == 0: whole groups of 4
          float gv[4];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int jj = j0 + j + k;
            const float x = __uint_as_float(v[j + k]) + (i == jj ? alpha : 0.f);
            gv[k] = zero ? 0.f : di * x * sd[jj];
          }
          *reinterpret_cast<float4 *>(p.G32 + o + j) = make_float4(gv[0], gv[1], gv[2], gv[3]);
          __nv_bfloat162 h0 = __floats2bfloat162_rn(gv[0], gv[1]);
          __nv_bfloat162 h1 = __floats2bfloat162_rn(gv[2], gv[3]);
          uint2 hv;
          hv.x = *reinterpret_cast<uint32_t *>(&h0);
          hv.y = *reinterpret_cast<uint32_t *>(&h1);
          *reinterpret_cast<uint2 *>(p.Ginv + o + j) = hv;
        }
      }
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 128);
  }
}

}  // namespace

cudaError_t launch_ns_fused(const CUtensorMap (&maps)[2][2], int batch, int r, int iters,
                            float ridge, const float *G, float *ex0, float *ex1, float *G32,
                            __nv_bfloat16 *Ginv, int *status, cudaStream_t s) {
  if (r <= 0 || r > kNsMaxR || r % 8 || iters <= 0) return cudaErrorInvalidValue;
  if (batch <= 0) return cudaSuccess;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(ns_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kNsfSmem);
  });
  if (attr_err != cudaSuccess) return attr_err;
  NsMaps m;
  for (int i = 0; i < 2; ++i)
    for (int j = 0; j < 2; ++j) m.m[i][j] = maps[i][j];
  NsParams p;
  p.r = r;
  p.rt = (r + 127) / 128;
  p.iters = iters;
  p.ridge = ridge;
  p.G = G;
  p.ex0 = ex0;
  p.ex1 = ex1;
  p.G32 = G32;
  p.Ginv = Ginv;
  p.status = status;
  p.idesc = tc_idesc(4, 0, 0, 128, 128);
  const unsigned nc = (unsigned)(2 * p.rt * p.rt);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2] = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = nc;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(nc, (unsigned)batch, 1);
  cfg.blockDim = dim3(kNsfThreads, 1, 1);
  cfg.dynamicSmemBytes = kNsfSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, ns_fused_kernel, m, p);
}

}  // namespace dyra
