// hyb_kernels.cu -- the hybrid ELL + dense-overflow activation format and its two
// training matmuls ("Sparser, Faster, Lighter Transformer Language Models",
// "Methodologie": rows with few nonzeros in a compact ELL matrix, rows with many in
// a dense backup matrix; hybrid-to-dense and dense-to-hybrid matrix multiplications
// for backpropagation).
//
// Layout (p24_hybrid in include/prune24.h): per row its nonzero count; ELL rows (at
// most E nonzeros) keep their nonzero columns ascending and their values, padded with
// column 0 / +0; overflow rows are numbered in row order and copied whole into the
// backup. A value is nonzero when its magnitude bits are not 0 (-0 is zero).
//
//  hyb_count_kernel   warp per row: counts nonzeros 8 values per lane (16-byte loads),
//                     places each one by a warp prefix sum and writes the ELL slots of
//                     rows that fit (a row that overflows has its slots cleared again).
//  hyb_scan_kernel    one CTA: numbers the overflow rows in row order (slot, list,
//                     count); more than the capacity sets P24_ECAPACITY in the status word.
//  hyb_copy_kernel    CTA per backup slot: copies the overflow row.
//  hyb_spmm_kernel    hybrid -> dense, Y = A B: CTA per (row, 2048 output columns);
//                     each nonzero (c, v) adds v * B[c, :] (one 16-byte row piece per
//                     thread, coalesced), fp32 accumulation, one rounding.
//  hyb_sddmm_kernel   dense -> hybrid, S = (G B^T) at A's nonzeros: CTA per row with
//                     G's row in shared memory; a warp per nonzero forms the dot product
//                     with B's row c and reduces it with shuffles.
// The overflow rows of both products go through the same loops: their nonzeros are
// first compacted, 2048 columns at a time, into the CTA's entry list.
//
// Bound: the products read one row of B (N bf16) per nonzero, mostly from L2; the
// count and copy kernels stream the dense input from HBM.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdint>

#include "p24_internal.h"

namespace p24 {
namespace {

__device__ __forceinline__ uint32_t nz_bits8(const uint4& x) {
  // bit i set where bf16 value i of the piece has nonzero magnitude bits
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t b = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    b |= ((w[i] & 0x7FFFu) != 0 ? 1u : 0u) << (2 * i);
    b |= ((w[i] & 0x7FFF0000u) != 0 ? 1u : 0u) << (2 * i + 1);
  }
  return b;
}

__device__ __forceinline__ uint16_t elem(const uint4& x, int j) {  // bf16 j (0..7) of the piece
  const uint32_t w = j < 4 ? (j < 2 ? x.x : x.y) : (j < 6 ? x.z : x.w);
  return static_cast<uint16_t>((j & 1) ? (w >> 16) : (w & 0xFFFFu));
}

// ---------------------------------------------------------------- format
__global__ void __launch_bounds__(256) hyb_count_kernel(const uint16_t* __restrict__ A, int64_t rows, int64_t cols,
                                                        int64_t lda, int E, int32_t* __restrict__ nnz,
                                                        uint16_t* __restrict__ ell_cols,
                                                        uint16_t* __restrict__ ell_vals) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const uint16_t* row = A + r * lda;
    uint16_t* oc = ell_cols + r * E;
    uint16_t* ov = ell_vals + r * E;
    int base = 0;  // nonzeros before this chunk of 256 columns
    for (int64_t c0 = 0; c0 < cols; c0 += 256) {
      const int64_t c = c0 + 8 * lane;
      uint4 x = make_uint4(0, 0, 0, 0);
      if (c < cols) x = __ldcs(reinterpret_cast<const uint4*>(row + c));  // cols % 8 == 0
      const uint32_t bits = nz_bits8(x);
      const int cnt = __popc(bits);
      int incl = cnt;  // inclusive prefix over the lanes
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
      }
      int pos = base + incl - cnt;
      if (pos < E) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (((bits >> j) & 1u) && pos < E) {
            oc[pos] = static_cast<uint16_t>(c + j);
            ov[pos] = elem(x, j);
          }
          pos += (bits >> j) & 1u;
        }
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    const int filled = base < E ? base : E;
    __syncwarp();
    // padding after the nonzeros; an overflow row (more than E) is cleared whole
    for (int i = (base > E ? 0 : filled) + lane; i < E; i += 32) {
      oc[i] = 0;
      ov[i] = 0;
    }
    if (lane == 0) nnz[r] = base;
  }
}

__global__ void __launch_bounds__(1024) hyb_scan_kernel(const int32_t* __restrict__ nnz, int64_t rows, int E,
                                                        int64_t cap, int32_t* __restrict__ slot,
                                                        int32_t* __restrict__ ovf_rows, int32_t* __restrict__ n_ovf,
                                                        int* status) {
  __shared__ int wsum[32];
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  int64_t offset = 0;
  for (int64_t r0 = 0; r0 < rows; r0 += 1024) {
    const int64_t r = r0 + t;
    const int f = (r < rows && nnz[r] > E) ? 1 : 0;
    int incl = f;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
      int v = wsum[lane];
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += y;
      }
      wsum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int64_t before = offset + (w > 0 ? wsum[w - 1] : 0) + incl - f;
    if (r < rows) {
      slot[r] = f ? static_cast<int32_t>(before) : -1;
      if (f && before < cap) ovf_rows[before] = static_cast<int32_t>(r);
    }
    offset += wsum[31];
    __syncthreads();
  }
  for (int64_t k = offset + t; k < cap; k += blockDim.x) ovf_rows[k] = -1;
  if (t == 0) {
    *n_ovf = static_cast<int32_t>(offset);
    if (offset > cap) atomicCAS(status, 0, -7 /* P24_ECAPACITY */);
  }
}

__global__ void __launch_bounds__(256) hyb_copy_kernel(const uint16_t* __restrict__ A, int64_t cols, int64_t lda,
                                                       const int32_t* __restrict__ ovf_rows,
                                                       const int32_t* __restrict__ n_ovf, int64_t cap,
                                                       uint16_t* __restrict__ ovf, int64_t ldo) {
  const int64_t k = blockIdx.x;
  const int64_t n = min(static_cast<int64_t>(*n_ovf), cap);
  if (k >= n) return;
  const uint16_t* src = A + static_cast<int64_t>(ovf_rows[k]) * lda;
  uint16_t* dst = ovf + k * ldo;
  for (int64_t c = 8 * static_cast<int64_t>(threadIdx.x); c < cols; c += 8 * blockDim.x)
    *reinterpret_cast<uint4*>(dst + c) = __ldcs(reinterpret_cast<const uint4*>(src + c));
}

// ---------------------------------------------------------------- products
constexpr int kHybChunk = 2048;  // backup columns compacted per round (8 per thread)

// Compacts the nonzeros of backup columns [c0, c0 + 2048) into (ecol, eval); returns
// their count (block-wide; every thread gets it). Column order is kept.
__device__ __forceinline__ int compact_chunk(const uint16_t* __restrict__ row, int64_t cols, int64_t c0,
                                             uint16_t* ecol, uint16_t* eval, int* wsum) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int64_t c = c0 + 8 * t;
  uint4 x = make_uint4(0, 0, 0, 0);
  if (c < cols) x = *reinterpret_cast<const uint4*>(row + c);
  const uint32_t bits = nz_bits8(x);
  const int cnt = __popc(bits);
  int incl = cnt;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += y;
  }
  __syncthreads();  // the previous round's entries are consumed
  if (lane == 31) wsum[w] = incl;
  __syncthreads();
  int before = incl - cnt;
  for (int i = 0; i < w; ++i) before += wsum[i];
  int total = 0;
  for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i) total += wsum[i];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if ((bits >> j) & 1u) {
      ecol[before] = static_cast<uint16_t>(c + j);
      eval[before] = elem(x, j);
      ++before;
    }
  }
  __syncthreads();
  return total;
}

// fp32 accumulation of n entries into 8 columns per thread: acc += v * B[c, n0 .. n0 + 7]
__device__ __forceinline__ void spmm_entries(const uint16_t* ecol, const uint16_t* eval, int n,
                                             const uint16_t* __restrict__ B, int64_t ldb, int64_t nb, bool ok,
                                             float (&acc)[8]) {
  int e = 0;
  for (; e + 4 <= n; e += 4) {
    uint4 b[4];
    float v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u] = __uint_as_float(static_cast<uint32_t>(eval[e + u]) << 16);
      b[u] = ok ? *reinterpret_cast<const uint4*>(B + static_cast<int64_t>(ecol[e + u]) * ldb + nb)
                : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = fmaf(v[u], __uint_as_float(static_cast<uint32_t>(elem(b[u], j)) << 16), acc[j]);
  }
  for (; e < n; ++e) {
    const float v = __uint_as_float(static_cast<uint32_t>(eval[e]) << 16);
    const uint4 b = ok ? *reinterpret_cast<const uint4*>(B + static_cast<int64_t>(ecol[e]) * ldb + nb)
                       : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(v, __uint_as_float(static_cast<uint32_t>(elem(b, j)) << 16), acc[j]);
  }
}

struct HybArgs {
  int64_t rows, cols, E, cap;
  const int32_t* nnz;
  const uint16_t* ell_cols;
  const uint16_t* ell_vals;
  const int32_t* slot;
  const uint16_t* ovf;
  int64_t ldo;
};

__global__ void __launch_bounds__(256) hyb_spmm_kernel(const HybArgs h, const uint16_t* __restrict__ B, int64_t N,
                                                       int64_t ldb, uint16_t* __restrict__ Y, int64_t ldy) {
  extern __shared__ uint16_t ent[];  // [max(E, 2048)] columns, then as many values
  __shared__ int wsum[32];
  const int64_t r = blockIdx.x;
  const int64_t ne = h.E > kHybChunk ? h.E : kHybChunk;
  uint16_t* ecol = ent;
  uint16_t* eval = ent + ne;
  const int64_t nb = static_cast<int64_t>(blockIdx.y) * 8 * blockDim.x + 8 * threadIdx.x;
  const bool ok = nb < N;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  const int s = h.slot[r];
  if (s < 0) {
    const int n = h.nnz[r];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      ecol[i] = h.ell_cols[r * h.E + i];
      eval[i] = h.ell_vals[r * h.E + i];
    }
    __syncthreads();
    spmm_entries(ecol, eval, n, B, ldb, nb, ok, acc);
  } else if (s < h.cap) {
    const uint16_t* row = h.ovf + static_cast<int64_t>(s) * h.ldo;
    for (int64_t c0 = 0; c0 < h.cols; c0 += kHybChunk) {
      const int n = compact_chunk(row, h.cols, c0, ecol, eval, wsum);
      spmm_entries(ecol, eval, n, B, ldb, nb, ok, acc);
    }
  }  // else: an overflow row past the capacity (P24_ECAPACITY is set): zeros
  if (ok) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * j], acc[2 * j + 1]);
      w[j] = *reinterpret_cast<uint32_t*>(&p);
    }
    *reinterpret_cast<uint4*>(Y + r * ldy + nb) = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// dot of G's staged row (bf16 in shared memory) with B's row c over N, one warp
__device__ __forceinline__ float warp_dot(const uint16_t* g, const uint16_t* __restrict__ brow, int64_t N) {
  const int lane = threadIdx.x & 31;
  float s = 0.f;
  for (int64_t n = 8 * lane; n < N; n += 256) {
    const uint4 b = *reinterpret_cast<const uint4*>(brow + n);
    const uint4 x = *reinterpret_cast<const uint4*>(g + n);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      s = fmaf(__uint_as_float(static_cast<uint32_t>(elem(x, j)) << 16),
               __uint_as_float(static_cast<uint32_t>(elem(b, j)) << 16), s);
  }
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) s += __shfl_xor_sync(0xffffffffu, s, d);
  return s;
}

__device__ __forceinline__ uint16_t to_bf16(float f) {
  __nv_bfloat16 b = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&b);
}

__global__ void __launch_bounds__(256) hyb_sddmm_kernel(const HybArgs h, const uint16_t* __restrict__ G, int64_t N,
                                                        int64_t ldg, const uint16_t* __restrict__ B, int64_t ldb,
                                                        uint16_t* __restrict__ S_ell, uint16_t* __restrict__ S_ovf,
                                                        int64_t lds) {
  extern __shared__ uint16_t sm[];  // G's row [N], then entry columns [max(E, 2048)]
  __shared__ int wsum[32];
  __shared__ uint16_t dummy_vals[kHybChunk];
  const int64_t r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  uint16_t* g = sm;
  uint16_t* ecol = sm + ((N + 7) / 8) * 8;
  for (int64_t n = 8 * threadIdx.x; n < N; n += 8 * blockDim.x)
    *reinterpret_cast<uint4*>(g + n) = *reinterpret_cast<const uint4*>(G + r * ldg + n);
  const int s = h.slot[r];
  if (s < 0) {
    const int n = h.nnz[r];
    for (int i = threadIdx.x; i < n; i += blockDim.x) ecol[i] = h.ell_cols[r * h.E + i];
    __syncthreads();
    for (int i = warp; i < n; i += nw) {
      const float d = warp_dot(g, B + static_cast<int64_t>(ecol[i]) * ldb, N);
      if (lane == 0) S_ell[r * h.E + i] = to_bf16(d);
    }
    for (int64_t i = n + threadIdx.x; i < h.E; i += blockDim.x) S_ell[r * h.E + i] = 0;
    return;
  }
  for (int64_t i = threadIdx.x; i < h.E; i += blockDim.x) S_ell[r * h.E + i] = 0;
  if (s >= h.cap) return;  // past the capacity (P24_ECAPACITY is set)
  const uint16_t* row = h.ovf + static_cast<int64_t>(s) * h.ldo;
  uint16_t* out = S_ovf + static_cast<int64_t>(s) * lds;
  for (int64_t c0 = 0; c0 < h.cols; c0 += kHybChunk) {
    // zeros for the chunk's columns, then the dots at its nonzeros (compact_chunk's
    // barriers order the two stores of a column)
    for (int64_t c = c0 + 8 * threadIdx.x; c < min(h.cols, c0 + kHybChunk); c += 8 * blockDim.x)
      *reinterpret_cast<uint4*>(out + c) = make_uint4(0, 0, 0, 0);
    __threadfence_block();
    const int n = compact_chunk(row, h.cols, c0, ecol, dummy_vals, wsum);
    for (int i = warp; i < n; i += nw) {
      const float d = warp_dot(g, B + static_cast<int64_t>(ecol[i]) * ldb, N);
      if (lane == 0) out[ecol[i]] = to_bf16(d);
    }
  }
}

HybArgs hyb_args(const p24_hybrid& h) {
  return HybArgs{h.rows,      h.cols, h.E, h.cap, h.nnz, h.ell_cols, static_cast<const uint16_t*>(h.ell_vals),
                 h.slot,      static_cast<const uint16_t*>(h.ovf), h.ldo};
}

}  // namespace

cudaError_t launch_hyb_compress(const void* A, int64_t lda, const p24_hybrid& h, int* status, cudaStream_t s) {
  if (h.rows == 0) return cudaSuccess;
  const auto* a = static_cast<const uint16_t*>(A);
  const int64_t blocks = std::min<int64_t>((h.rows + 7) / 8, 152 * 32);
  hyb_count_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a, h.rows, h.cols, lda, static_cast<int>(h.E), h.nnz,
                                                                 h.ell_cols, static_cast<uint16_t*>(h.ell_vals));
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  hyb_scan_kernel<<<1, 1024, 0, s>>>(h.nnz, h.rows, static_cast<int>(h.E), h.cap, h.slot, h.ovf_rows, h.n_ovf,
                                     status);
  count_launch();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if (h.cap > 0) {
    hyb_copy_kernel<<<static_cast<unsigned>(h.cap), 256, 0, s>>>(a, h.cols, lda, h.ovf_rows, h.n_ovf, h.cap,
                                                                 static_cast<uint16_t*>(h.ovf), h.ldo);
    count_launch();
  }
  return cudaGetLastError();
}

cudaError_t launch_hyb_spmm(const p24_hybrid& h, const void* B, int64_t N, int64_t ldb, void* Y, int64_t ldy,
                            cudaStream_t s) {
  if (h.rows == 0 || N == 0) return cudaSuccess;
  const int64_t ne = std::max<int64_t>(h.E, kHybChunk);
  const size_t smem = static_cast<size_t>(ne) * 4;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(hyb_spmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  dim3 grid(static_cast<unsigned>(h.rows), static_cast<unsigned>((N + 2047) / 2048));
  hyb_spmm_kernel<<<grid, 256, smem, s>>>(hyb_args(h), static_cast<const uint16_t*>(B), N, ldb,
                                          static_cast<uint16_t*>(Y), ldy);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_hyb_sddmm(const p24_hybrid& h, const void* G, int64_t N, int64_t ldg, const void* B, int64_t ldb,
                             void* S_ell, void* S_ovf, int64_t lds, cudaStream_t s) {
  if (h.rows == 0) return cudaSuccess;
  const int64_t ne = std::max<int64_t>(h.E, kHybChunk);
  const size_t smem = static_cast<size_t>((N + 7) / 8 * 8 + ne) * 2;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(hyb_sddmm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  hyb_sddmm_kernel<<<static_cast<unsigned>(h.rows), 256, smem, s>>>(
      hyb_args(h), static_cast<const uint16_t*>(G), N, ldg, static_cast<const uint16_t*>(B), ldb,
      static_cast<uint16_t*>(S_ell), static_cast<uint16_t*>(S_ovf), lds);
  count_launch();
  return cudaGetLastError();
}

}  // namespace p24
