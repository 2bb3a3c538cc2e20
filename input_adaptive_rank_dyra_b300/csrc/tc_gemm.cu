// Persistent TMA + tcgen05 GEMM engine used by every dense contraction of the bf16 DyRA
// forward. See tc_gemm.cuh for the roles of the warps and the epilogue modes.
#include "tc_gemm.cuh"
#include "ptx.cuh"

#include <cuda_bf16.h>
#include <mutex>

namespace dyra {

namespace {

constexpr uint32_t kStagingBytesPerWarp = 2 * 2048;   // two 32 x 32 bf16 buffers

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Row of 16 fp32 values -> bf16, written with two 16-byte stores when in range and aligned.
__device__ __forceinline__ void store_row16_bf16(__nv_bfloat16 *dst, const float *f, int valid) {
  if (valid >= 16 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
    uint4 w0 = make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                          pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
    uint4 w1 = make_uint4(pack_bf16x2(f[8], f[9]), pack_bf16x2(f[10], f[11]),
                          pack_bf16x2(f[12], f[13]), pack_bf16x2(f[14], f[15]));
    reinterpret_cast<uint4 *>(dst)[0] = w0;
    reinterpret_cast<uint4 *>(dst)[1] = w1;
  } else {
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < valid) dst[j] = __float2bfloat16_rn(f[j]);
  }
}

struct TileCoord {
  int bz, m_tile, n_tile;
};

__device__ __forceinline__ TileCoord decode_tile(int t, const TcGemmParams &p) {
  TileCoord c;
  c.n_tile = t % p.n_tiles;
  const int rest = t / p.n_tiles;
  c.m_tile = rest % p.m_tiles;
  c.bz = rest / p.m_tiles;
  return c;
}

// Epilogue of 16 accumulator columns [col0, col0 + 16) of row g, direct global stores.
__device__ __forceinline__ void epilogue16(const TcGemmParams &p, const float *f, long long g,
                                           int col0, int bz, bool second) {
  const int cols_lim = (p.epi == EPI_CG && second) ? p.cols2_valid : p.cols_valid;
  const int valid = cols_lim - col0;
  if (valid <= 0) return;
  if (p.epi == EPI_ROW_BF16) {
    if (g < p.rows_valid) {
      float h[16];
#pragma unroll
      for (int j = 0; j < 16; ++j)
        h[j] = f[j] + ((p.bias && j < valid) ? __ldg(p.bias + col0 + j) : 0.f);
      __nv_bfloat16 *dst =
          reinterpret_cast<__nv_bfloat16 *>(p.out) + bz * p.out_bstride + g * p.out_ld + col0;
      store_row16_bf16(dst, h, valid);
    }
  } else if (p.epi == EPI_TRANS_BF16) {
    if (g < p.rows_valid) {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + bz * p.out_bstride +
                           (g / p.rb) * p.out_gstride + (g % p.rb);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < valid) dst[(long long)(col0 + j) * p.out_ld] = __float2bfloat16_rn(f[j]);
    }
  } else if (p.epi == EPI_CG) {
    if (!second) {
      if (g < p.rows_valid) {
        __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + bz * p.out_bstride + g;
#pragma unroll
        for (int j = 0; j < 16; ++j)
          if (j < valid) dst[(long long)(col0 + j) * p.out_ld] = __float2bfloat16_rn(f[j]);
      }
    } else if (g < p.rows2_valid) {
      float *dst = reinterpret_cast<float *>(p.out2) + bz * p.out2_bstride + g * p.out2_ld + col0;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < valid) dst[j] = f[j];
    }
  } else if (p.epi == EPI_TRANS_F32) {
    if (g < p.rows_valid) {
      float *dst = reinterpret_cast<float *>(p.out) + bz * p.out_bstride +
                   (g / p.rb) * p.out_gstride + (g % p.rb);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < valid) dst[(long long)(col0 + j) * p.out_ld] = p.alpha * f[j];
    }
  } else {   // EPI_ROW_F32
    if (g < p.rows_valid) {
      float *dst = reinterpret_cast<float *>(p.out) + bz * p.out_bstride + g * p.out_ld + col0;
      const float *ax = p.aux ? p.aux + bz * p.aux_bstride + g * p.aux_ld + col0 : nullptr;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        if (j < valid) dst[j] = p.alpha * f[j] + (ax ? p.beta * ax[j] : 0.f);
    }
  }
}

__global__ void __launch_bounds__(192, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
                   const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                   const __grid_constant__ CUtensorMap tmOut, const __grid_constant__ TcGemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (base - raw_addr);
  const int S = p.stages;
  const uint32_t a_bytes = 16384u;
  const uint32_t b_bytes = (uint32_t)p.BN * 128u;
  const uint32_t stage_bytes = a_bytes + b_bytes;
  const uint32_t staging = base + p.staging_off;
  const uint32_t bar_base = staging + (p.tma_store ? 4u * kStagingBytesPerWarp : 0u);
  // full[S] | empty[S] | tfull[2] | tempty[2] | tmem slot
  const uint32_t full_bar = bar_base, empty_bar = bar_base + 8u * S;
  const uint32_t tfull_bar = bar_base + 16u * S, tempty_bar = tfull_bar + 16u;
  const uint32_t tmem_slot = tempty_bar + 16u;
  volatile uint32_t *tmem_slot_ptr =
      reinterpret_cast<volatile uint32_t *>(smem + (tmem_slot - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = 128 / p.elem_bytes;   // elements in one 128-byte row
  const int total = p.batch * p.m_tiles * p.n_tiles;

  if (warp == 0 && lane == 0) {
    for (int s = 0; s < S; ++s) {
      ptx::mbar_init(full_bar + 8u * s, 1);
      ptx::mbar_init(empty_bar + 8u * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(tfull_bar + 8u * a, 1);
      ptx::mbar_init(tempty_bar + 8u * a, 4);   // one arrival per epilogue warp
    }
    ptx::mbar_init_fence();
    ptx::tma_prefetch_desc(&tmA0);
    ptx::tma_prefetch_desc(&tmB0);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tmem_slot, 2u * p.acc_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot_ptr;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t q = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile(t, p);
        const bool a_second = tc.m_tile >= p.a_split;
        const int m0 = (a_second ? tc.m_tile - p.a_split : tc.m_tile) * 128;
        const int n0 = tc.n_tile * p.BN;
        const CUtensorMap *ma = a_second ? &tmA1 : &tmA0;
        const int a_b = (a_second ? p.a_batched1 : p.a_batched0) ? tc.bz : 0;
        for (int kc = 0; kc < p.k_chunks; ++kc, ++q) {
          const uint32_t s = q % (uint32_t)S;
          const uint32_t round = q / (uint32_t)S;
          if (!ptx::mbar_wait(empty_bar + 8u * s, (round & 1u) ^ 1u, p.timeouts)) {
            ok = false;
            break;
          }
          const uint32_t full = full_bar + 8u * s;
          ptx::mbar_arrive_expect_tx(full, stage_bytes);
          const uint32_t sa = base + s * stage_bytes, sb = sa + a_bytes;
          if (p.a_major == 0) {
            ptx::tma_load_3d(sa, ma, full, kc * chunk, m0, a_b);
          } else {
            for (int i = 0; i < 128 / chunk; ++i)
              ptx::tma_load_3d(sa + (uint32_t)(i * chunk * 128), ma, full, m0 + i * chunk,
                               kc * chunk, a_b);
          }
          const bool b_second = kc >= p.b_split;
          const CUtensorMap *mb = b_second ? &tmB1 : &tmB0;
          const int kk = b_second ? kc - p.b_split : kc;
          const int b_b = (b_second ? p.b_batched1 : p.b_batched0) ? tc.bz : 0;
          if (p.b_major == 0) {
            ptx::tma_load_3d(sb, mb, full, kk * chunk, n0, b_b);
          } else {
            for (int i = 0; i < p.BN / chunk; ++i)
              ptx::tma_load_3d(sb + (uint32_t)(i * chunk * 128), mb, full, n0 + i * chunk,
                               kk * chunk, b_b);
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      // K-major SW128: rows of 128 B, 8-row groups 1024 B apart (SBO), K advance inside the row.
      // MN-major SW128: 128-byte rows hold `chunk` MN elements; MN groups LBO apart, 8-row K
      // groups 1024 B apart; one MMA consumes 32 bytes of K = 32/elem rows.
      const uint32_t a_lbo = p.a_major ? (uint32_t)(chunk * 128) : 16u;
      const uint32_t b_lbo = p.b_major ? (uint32_t)(chunk * 128) : 16u;
      const uint32_t a_kstep = p.a_major ? 4096u / (uint32_t)p.elem_bytes : 32u;
      const uint32_t b_kstep = p.b_major ? 4096u / (uint32_t)p.elem_bytes : 32u;
      uint32_t q = 0, i = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++i) {
        const uint32_t acc = i & 1u;
        if (!ptx::mbar_wait(tempty_bar + 8u * acc, ((i >> 1) & 1u) ^ 1u, p.timeouts)) break;
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * p.acc_cols;
        for (int kc = 0; kc < p.k_chunks; ++kc, ++q) {
          const uint32_t s = q % (uint32_t)S;
          const uint32_t round = q / (uint32_t)S;
          if (!ptx::mbar_wait(full_bar + 8u * s, round & 1u, p.timeouts)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t sa = base + s * stage_bytes, sb = sa + a_bytes;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = ptx::sdesc_sw128(sa + ks * a_kstep, a_lbo, 1024u);
            const uint64_t bd = ptx::sdesc_sw128(sb + ks * b_kstep, b_lbo, 1024u);
            const uint32_t accum = (kc | ks) ? 1u : 0u;
            if (p.elem_bytes == 2)
              ptx::tc_mma_f16(d_tmem, ad, bd, p.idesc, accum);
            else
              ptx::tc_mma_tf32(d_tmem, ad, bd, p.idesc, accum);
          }
          ptx::tc_commit(empty_bar + 8u * s);   // frees the smem stage when these MMAs finish
        }
        if (ok) ptx::tc_commit(tfull_bar + 8u * acc);   // accumulator ready
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;   // TMEM lane quarter this warp may read
    const uint32_t stg = staging + (uint32_t)(warp - 2) * kStagingBytesPerWarp;
    uint32_t buf = 0, i = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++i) {
      const uint32_t acc = i & 1u;
      int got = 0;
      if (lane == 0) got = ptx::mbar_wait(tfull_bar + 8u * acc, (i >> 1) & 1u, p.timeouts) ? 1 : 0;
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      ptx::tc_fence_after();
      const TileCoord tc = decode_tile(t, p);
      const bool second = tc.m_tile >= p.a_split;
      const int m0 = (second ? tc.m_tile - p.a_split : tc.m_tile) * 128;
      const int n0 = tc.n_tile * p.BN;
      const uint32_t taddr = tmem_base + acc * p.acc_cols + ((uint32_t)(q * 32) << 16);
      const long long g = (long long)m0 + q * 32 + lane;
      const int cols_lim = (p.epi == EPI_CG && second) ? p.cols2_valid : p.cols_valid;
      if (p.tma_store) {
        // bf16 rows through a 64B-swizzled 32 x 32 staging tile and a TMA bulk store
        const int row0 = m0 + q * 32;
        for (int c0 = 0; c0 < p.BN; c0 += 32) {
          const int col0 = n0 + c0;
          if (col0 >= cols_lim) break;   // uniform across the warp
          uint32_t v[32];
          ptx::tmem_ld32(taddr + (uint32_t)c0, v);
          ptx::tmem_ld_wait();
          if (row0 >= p.rows_valid) continue;   // whole 32-row slab outside the tensor
          float f[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            f[j] = __uint_as_float(v[j]);
            if (p.bias && col0 + j < cols_lim) f[j] += __ldg(p.bias + col0 + j);
          }
          if (lane == 0) ptx::bulk_wait_read<1>();   // this buffer's previous store has read it
          __syncwarp();
          const uint32_t dst = stg + buf * 2048u + (uint32_t)lane * 64u;
          const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint32_t w0 = pack_bf16x2(f[8 * c + 0], f[8 * c + 1]);
            const uint32_t w1 = pack_bf16x2(f[8 * c + 2], f[8 * c + 3]);
            const uint32_t w2 = pack_bf16x2(f[8 * c + 4], f[8 * c + 5]);
            const uint32_t w3 = pack_bf16x2(f[8 * c + 6], f[8 * c + 7]);
            const uint32_t addr = dst + (((uint32_t)c ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1),
                         "r"(w2), "r"(w3)
                         : "memory");
          }
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            ptx::tma_store_3d(&tmOut, stg + buf * 2048u, col0, row0, p.out_batched ? tc.bz : 0);
            ptx::bulk_commit();
          }
          buf ^= 1u;
        }
      } else {
        for (int c0 = 0; c0 < p.BN; c0 += 32) {
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
      if (lane == 0) ptx::mbar_arrive(tempty_bar + 8u * acc);
    }
    if (p.tma_store && lane == 0) ptx::bulk_wait<0>();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
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

uint32_t tc_idesc(int elem_bytes, int a_major, int b_major, int n) {
  const uint32_t fmt = elem_bytes == 2 ? 1u : 2u;   // BF16 = 1, TF32 = 2
  uint32_t d = 0;
  d |= 1u << 4;                          // D format: F32
  d |= fmt << 7;                         // A format
  d |= fmt << 10;                        // B format
  d |= (uint32_t)(a_major & 1) << 15;    // A major (1 = MN)
  d |= (uint32_t)(b_major & 1) << 16;    // B major
  d |= ((uint32_t)n >> 3) << 17;         // N / 8
  d |= (128u >> 4) << 24;                // M / 16
  return d;
}

bool tc_make_map(CUtensorMap *map, const TcOperand &op, int box_rows) {
  return encode(map, op, (cuuint32_t)(128 / op.elem_bytes), (cuuint32_t)box_rows,
                CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tc_make_store_map(CUtensorMap *map, const TcOperand &op) {
  return encode(map, op, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}

cudaError_t tc_gemm_launch(TcGemmParams p, const CUtensorMap &a0, const CUtensorMap &a1,
                           const CUtensorMap &b0, const CUtensorMap &b1,
                           const CUtensorMap &out_map, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, []() {
    attr_err = cudaFuncSetAttribute(tc_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    232448);
  });
  if (attr_err != cudaSuccess) return attr_err;
  if (p.m_tiles <= 0 || p.n_tiles <= 0 || p.batch <= 0 || p.k_chunks <= 0) return cudaSuccess;
  // MN-major tf32 operands need the 32-byte-atom 128B swizzle, which this engine does not
  // set up; every tf32 use here is K-major.
  if (p.elem_bytes == 4 && (p.a_major || p.b_major)) return cudaErrorNotSupported;
  if (p.BN < 16 || p.BN > 256 || p.BN % 16) return cudaErrorInvalidValue;
  if (p.tma_store && (p.epi != EPI_ROW_BF16 || p.BN % 32)) return cudaErrorInvalidValue;
  p.acc_cols = 32;
  while (p.acc_cols < (uint32_t)p.BN) p.acc_cols <<= 1;
  const uint32_t stage = 16384u + (uint32_t)p.BN * 128u;
  const uint32_t staging = p.tma_store ? 4u * kStagingBytesPerWarp : 0u;
  const uint32_t fixed = 1024u + staging + 256u;   // alignment slack, staging, barriers
  int S = (int)((232448u - fixed) / stage);
  if (S > 8) S = 8;
  if (S < 2) return cudaErrorInvalidValue;
  p.stages = S;
  p.staging_off = (uint32_t)S * stage;
  uint32_t smem = (uint32_t)S * stage + fixed;
  // one CTA per SM: the two accumulators may take all 512 TMEM columns
  if (smem < 116u * 1024u) smem = 116u * 1024u;
  p.smem_bytes = smem;
  const long long total = (long long)p.batch * p.m_tiles * p.n_tiles;
  const int grid = (int)(total < num_sms() ? total : num_sms());
  tc_gemm_kernel<<<grid, 192, smem, stream>>>(a0, a1, b0, b1, out_map, p);
  return cudaGetLastError();
}

}  // namespace dyra
