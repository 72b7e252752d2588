// prune24_kernels.cu -- HBM-bound kernels of the 2:4 path: magnitude pruning
// + compression, the double prune of the transposed weight, padding of
// compressed rows, and deterministic column sums (bias gradients).
//
// Method (inno4scale "Success story ESPLAG", "Solution": N:M pruning with a
// compressed storage format; SLOPE abstract, NSF PAR award 2340011: the
// transposed weight is pruned again with N:M for the backward pass):
// in each group of 4 consecutive values the two of largest magnitude are kept;
// magnitude = bf16 bits with the sign cleared; ties go to the lower index.
// Every decision is integer, so the outputs are a pure function of the input bits.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "p24_internal.h"
#include "p24_ptx.cuh"

namespace p24 {
namespace {

// ---------------------------------------------------------------- the 2:4 pick
// A group of four bf16 values is held as two 32-bit words: lo = e0 | e1 << 16,
// hi = e2 | e3 << 16. Each value gets a composite key (magnitude << 2) | (3 - i):
// distinct for the four positions, larger = kept first, and among equal
// magnitudes the lower index has the larger key. The two largest composites
// come out of a 4-input max/min network.
__device__ __forceinline__ uint32_t pick2_nibble(uint32_t lo, uint32_t hi) {
  const uint32_t c0 = ((lo & 0x7FFFu) << 2) | 3u;
  const uint32_t c1 = ((lo >> 14) & 0x1FFFCu) | 2u;
  const uint32_t c2 = ((hi & 0x7FFFu) << 2) | 1u;
  const uint32_t c3 = (hi >> 14) & 0x1FFFCu;
  const uint32_t a = max(c0, c1), b = min(c0, c1);
  const uint32_t c = max(c2, c3), d = min(c2, c3);
  const uint32_t top = max(a, c);
  const uint32_t second = max(min(a, c), max(b, d));
  const uint32_t i_top = 3u - (top & 3u), i_sec = 3u - (second & 3u);
  return min(i_top, i_sec) | (max(i_top, i_sec) << 2);
}

// The same network, returning which two positions won as a 4-bit code
// (3 - i_top) << 2 | (3 - i_sec): the row of a 16-entry table (pick_row) that holds
// everything the caller derives from the decision. Here the composite keys are
// (magnitude << 17) | (3 - i): multiplying a 16-bit value by 2^17 drops its sign
// bit and everything above it, so each key is one multiply-add (and a shift for
// the upper half), which keeps the integer ALU pipe free for the min/max network.
__device__ __forceinline__ uint32_t pick2_code(uint32_t lo, uint32_t hi) {
  const uint32_t c0 = lo * 131072u + 3u;
  const uint32_t c1 = (lo >> 16) * 131072u + 2u;
  const uint32_t c2 = hi * 131072u + 1u;
  const uint32_t c3 = (hi >> 16) * 131072u;
  const uint32_t a = max(c0, c1), b = min(c0, c1);
  const uint32_t c = max(c2, c3), d = min(c2, c3);
  const uint32_t top = max(a, c);
  const uint32_t second = max(min(a, c), max(b, d));
  return ((top & 3u) << 2) | (second & 3u);
}

// pick2_code with the upper halves taken by a multiply-high (hi16 = 2^16, passed at
// run time so that it stays a multiply): the shift moves from the integer pipe to the
// FMA pipe, which the prune kernels leave mostly idle.
__device__ __forceinline__ uint32_t pick2_code_mh(uint32_t lo, uint32_t hi, uint32_t hi16) {
  const uint32_t c0 = lo * 131072u + 3u;
  const uint32_t c1 = __umulhi(lo, hi16) * 131072u + 2u;
  const uint32_t c2 = hi * 131072u + 1u;
  const uint32_t c3 = __umulhi(hi, hi16) * 131072u;
  const uint32_t a = max(c0, c1), b = min(c0, c1);
  const uint32_t c = max(c2, c3), d = min(c2, c3);
  const uint32_t top = max(a, c);
  const uint32_t second = max(min(a, c), max(b, d));
  return ((top & 3u) << 2) | (second & 3u);
}

// Row of the pick table for code t (unused codes, where both positions agree, are 0):
//   x = byte selector of the kept pair from (lo, hi) | nibble << 16
//   y = selector keeping lo's kept halves (others from a zero word) | the same for hi << 16
// A prmt reads only the low 16 bits of its selector.
__device__ __forceinline__ uint2 pick_row(uint32_t t) {
  const uint32_t it = 3u - (t >> 2), is = 3u - (t & 3u);
  if (it == is) return make_uint2(0u, 0u);
  const uint32_t i0 = min(it, is), i1 = max(it, is);
  const uint32_t kb = (1u << i0) | (1u << i1);
  const uint32_t sel_kept = 0x1010u + i0 * 0x22u + i1 * 0x2200u;
  const uint32_t mlo = ((kb & 1u) ? 0x0010u : 0x0044u) | ((kb & 2u) ? 0x3200u : 0x4400u);
  const uint32_t mhi = ((kb & 4u) ? 0x0010u : 0x0044u) | ((kb & 8u) ? 0x3200u : 0x4400u);
  return make_uint2(sel_kept | ((i0 | (i1 << 2)) << 16), mlo | (mhi << 16));
}

// The two kept values (ascending index) packed as v0 | v1 << 16.
__device__ __forceinline__ uint32_t kept_pair(uint32_t lo, uint32_t hi, uint32_t nib) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  const uint32_t sel = 0x1010u + i0 * 0x22u + i1 * 0x2200u;  // bytes 2i0,2i0+1,2i1,2i1+1
  return __byte_perm(lo, hi, sel);
}

// The group with its dropped values set to +0.
__device__ __forceinline__ void masked_group(uint32_t lo, uint32_t hi, uint32_t nib, uint32_t& mlo,
                                             uint32_t& mhi) {
  const uint32_t kb = (1u << (nib & 3u)) | (1u << (nib >> 2));
  mlo = lo & (((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u));
  mhi = hi & (((kb & 4u) ? 0x0000FFFFu : 0u) | ((kb & 8u) ? 0xFFFF0000u : 0u));
}

// Scatter two kept values back into a dense group.
__device__ __forceinline__ void expand_group(uint32_t pair, uint32_t nib, uint32_t& lo, uint32_t& hi) {
  const uint32_t i0 = nib & 3u, i1 = (nib >> 2) & 3u;
  const uint64_t v = (static_cast<uint64_t>(pair & 0xFFFFu) << (16u * i0)) |
                     (static_cast<uint64_t>(pair >> 16) << (16u * i1));
  lo = static_cast<uint32_t>(v);
  hi = static_cast<uint32_t>(v >> 32);
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

// ---------------------------------------------------------------- compress
// One thread = one 16-byte piece (8 values, 2 groups) per step; a CTA of 256
// threads covers 1024 consecutive pieces of a row, 4 per thread, loads first.
template <bool kMasked>
__global__ void __launch_bounds__(256) compress_kernel(const uint16_t* __restrict__ W, int64_t rows, int64_t cols,
                                                       int64_t ldw, uint16_t* __restrict__ vals, int64_t ldv,
                                                       uint8_t* __restrict__ meta, int64_t ldm,
                                                       uint16_t* __restrict__ Wm, int64_t ldwm) {
  for (int64_t row = blockIdx.y; row < rows; row += gridDim.y) {
    const uint16_t* w = W + row * ldw;
    const int64_t p0 = static_cast<int64_t>(blockIdx.x) * 1024 + threadIdx.x;
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t e = (p0 + j * 256) * 8;
      v[j] = make_uint4(0, 0, 0, 0);
      if (e + 8 <= cols) {
        v[j] = ld_stream_v4(w + e);
      } else if (e + 4 <= cols) {
        const uint2 h = __ldcs(reinterpret_cast<const uint2*>(w + e));
        v[j].x = h.x;
        v[j].y = h.y;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t p = p0 + j * 256;
      const int64_t e = p * 8;
      if (e + 4 > cols) continue;
      const uint32_t n0 = pick2_nibble(v[j].x, v[j].y);
      const uint32_t k0 = kept_pair(v[j].x, v[j].y, n0);
      if (e + 8 <= cols) {
        const uint32_t n1 = pick2_nibble(v[j].z, v[j].w);
        const uint32_t k1 = kept_pair(v[j].z, v[j].w, n1);
        *reinterpret_cast<uint2*>(vals + row * ldv + p * 4) = make_uint2(k0, k1);
        meta[row * ldm + p] = static_cast<uint8_t>(n0 | (n1 << 4));
        if (kMasked) {
          uint4 m;
          masked_group(v[j].x, v[j].y, n0, m.x, m.y);
          masked_group(v[j].z, v[j].w, n1, m.z, m.w);
          *reinterpret_cast<uint4*>(Wm + row * ldwm + e) = m;
        }
      } else {
        *reinterpret_cast<uint32_t*>(vals + row * ldv + p * 4) = k0;
        meta[row * ldm + p] = static_cast<uint8_t>(n0 | 0x40u);  // odd group count: pad high nibble
        if (kMasked) {
          uint2 m;
          masked_group(v[j].x, v[j].y, n0, m.x, m.y);
          *reinterpret_cast<uint2*>(Wm + row * ldwm + e) = m;
        }
      }
    }
  }
}

// ---------------------------------------------------------------- V:2:M prune
// Vector-wise N:M (the VENOM format of the ESPLAG success story, "Solution"; v:n:m
// activations in the TO24 abstract): in every block of V rows and group of M
// columns the same 4 columns are kept for all rows of the block (the 4 largest
// L1 norms over the block, ties to the lower column), then each row keeps 2 of
// those 4 by the 2:4 rule. Output: the selected column offsets, and the condensed
// [rows, 4 cols / M] matrix in the 2:4 format.
//
// A CTA owns one block of rows and 256 consecutive columns (M divides 256, so
// groups never straddle CTAs, and with M <= 128 a CTA holds whole pairs of groups,
// i.e. whole metadata bytes).
//   1. thread = column: its L1 norm over the block, fp32, rows in order; the
//      ranking key is the sum's bit pattern (every NaN as 0x7FC00000);
//   2. thread = column: kept iff fewer than 4 columns of its group beat it
//      (larger key, or equal key and lower column); its rank among the kept
//      columns of the group gives its slot in the ascending offset list;
//   3. threads = (row, pair of groups): the 4 values at the kept columns are
//      pruned 2:4 and written as values plus one metadata byte.
constexpr int kVnmCols = 256;

__global__ void __launch_bounds__(256) vnm_compress_kernel(const uint16_t* __restrict__ A, int64_t rows,
                                                           int64_t cols, int64_t lda, int V, int M,
                                                           uint8_t* __restrict__ colidx, uint16_t* __restrict__ vals,
                                                           int64_t ldv, uint8_t* __restrict__ meta, int64_t ldm) {
  __shared__ uint32_t key[kVnmCols];
  __shared__ uint8_t kept[kVnmCols];
  __shared__ uint8_t offs[kVnmCols];  // [group in chunk][slot 0..3]: up to 64 groups of 4
  const int t = threadIdx.x;
  const int64_t G = cols / M;                    // groups per row
  const int64_t nb = (rows + V - 1) / V;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * kVnmCols;
  const int64_t c = c0 + t;
  const int j = t % M, gstart = t - j;           // column within its group, group's first thread
  const int gpc = kVnmCols / M;                  // groups per chunk (even: M <= 128)
  for (int64_t b = blockIdx.y; b < nb; b += gridDim.y) {
    const int64_t r0 = b * V;
    const int64_t r1 = min(rows, r0 + V);
    // 1. column norm over the block
    float sum = 0.f;
    if (c < cols)
      for (int64_t r = r0; r < r1; ++r) sum += __uint_as_float(static_cast<uint32_t>(A[r * lda + c] & 0x7FFFu) << 16);
    const uint32_t k = (sum != sum) ? 0x7FC00000u : __float_as_uint(sum);
    key[t] = k;
    __syncthreads();
    // 2. selection and slot
    int beat = 0;
    for (int q = 0; q < M; ++q) {
      const uint32_t kq = key[gstart + q];
      beat += (kq > k || (kq == k && q < j)) ? 1 : 0;
    }
    kept[t] = beat < 4 ? 1 : 0;
    __syncthreads();
    if (kept[t]) {
      int slot = 0;
      for (int q = 0; q < j; ++q) slot += kept[gstart + q];
      offs[(t / M) * 4 + slot] = static_cast<uint8_t>(j);
      if (c < cols) colidx[(b * G + c / M) * 4 + slot] = static_cast<uint8_t>(j);
    }
    __syncthreads();
    // 3. rows of the block x pairs of groups of the chunk
    const int pairs = gpc / 2;
    const int64_t g_first = c0 / M;              // even
    const int64_t nwork = (r1 - r0) * pairs;
    for (int64_t w = t; w < nwork; w += blockDim.x) {
      const int64_t r = r0 + w / pairs;
      const int pl = static_cast<int>(w % pairs);
      uint32_t nib[2] = {0x4u, 0x4u};
      for (int h = 0; h < 2; ++h) {
        const int gl = 2 * pl + h;               // group within the chunk
        const int64_t gg = g_first + gl;         // group within the row
        if (gg >= G) break;
        const uint16_t* a = A + r * lda + gg * M;
        const uint8_t* o = offs + gl * 4;
        const uint32_t lo = static_cast<uint32_t>(a[o[0]]) | (static_cast<uint32_t>(a[o[1]]) << 16);
        const uint32_t hi = static_cast<uint32_t>(a[o[2]]) | (static_cast<uint32_t>(a[o[3]]) << 16);
        nib[h] = pick2_nibble(lo, hi);
        *reinterpret_cast<uint32_t*>(vals + r * ldv + 2 * gg) = kept_pair(lo, hi, nib[h]);
      }
      if (g_first + 2 * pl < G) meta[r * ldm + (g_first + 2 * pl) / 2] = static_cast<uint8_t>(nib[0] | (nib[1] << 4));
    }
    __syncthreads();
  }
}

// The same prune with the CTA's block (V <= 256 rows x CW columns) staged in shared
// memory: one coalesced pass of 16-byte loads brings the block on chip, the column
// norms (same fp32 order: rows of the block top to bottom), the selection and the
// row prunes then read shared memory, and the optional dense masked output is
// written back from it with 16-byte stores. The whole block is read before anything
// is written, so the masked output may overwrite A in place.
// CW = 64 for M <= 32, else 2 M (CW / M is even, so whole metadata bytes fall in one CTA).
__global__ void __launch_bounds__(256) vnm_compress_staged_kernel(
    const uint16_t* A, int64_t rows, int64_t cols, int64_t lda, int V, int M, int CW,
    uint8_t* __restrict__ colidx, uint16_t* __restrict__ vals, int64_t ldv, uint8_t* __restrict__ meta, int64_t ldm,
    uint16_t* Am, int64_t ldam) {
  extern __shared__ __align__(16) uint16_t tile[];  // [V][CW]
  __shared__ uint32_t key[256];
  __shared__ uint8_t kept[256];
  __shared__ uint8_t offs[256];  // [group in chunk][slot 0..3]
  const int t = threadIdx.x;
  const int64_t G = cols / M;
  const int64_t nb = (rows + V - 1) / V;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * CW;
  const int ncol = static_cast<int>(min(static_cast<int64_t>(CW), cols - c0));  // a multiple of M and of 8
  const int cpr = ncol / 8;                       // 16-byte chunks per row
  const int j = t % M, gstart = t - j;            // column within its group, group's first column
  const int gpc = ncol / M;                       // groups in this chunk (odd only in a row's last chunk)
  for (int64_t b = blockIdx.y; b < nb; b += gridDim.y) {
    const int64_t r0 = b * V;
    const int nr = static_cast<int>(min(rows - r0, static_cast<int64_t>(V)));
    // 1. stage the block
    const int nchunks = nr * cpr;
    for (int i0 = t; i0 < nchunks; i0 += 4 * 256) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 256;
        if (i < nchunks) v[u] = ld_stream_v4(A + (r0 + i / cpr) * lda + c0 + (i % cpr) * 8);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int i = i0 + u * 256;
        if (i < nchunks) *reinterpret_cast<uint4*>(tile + (i / cpr) * CW + (i % cpr) * 8) = v[u];
      }
    }
    __syncthreads();
    // 2. column norm over the block, rows in order
    if (t < ncol) {
      float sum = 0.f;
      for (int r = 0; r < nr; ++r) sum += __uint_as_float(static_cast<uint32_t>(tile[r * CW + t] & 0x7FFFu) << 16);
      key[t] = (sum != sum) ? 0x7FC00000u : __float_as_uint(sum);
    }
    __syncthreads();
    // 3. selection and slot
    if (t < ncol) {
      const uint32_t k = key[t];
      int beat = 0;
      for (int q = 0; q < M; ++q) {
        const uint32_t kq = key[gstart + q];
        beat += (kq > k || (kq == k && q < j)) ? 1 : 0;
      }
      kept[t] = beat < 4 ? 1 : 0;
    }
    __syncthreads();
    if (t < ncol && kept[t]) {
      int slot = 0;
      for (int q = 0; q < j; ++q) slot += kept[gstart + q];
      offs[(t / M) * 4 + slot] = static_cast<uint8_t>(j);
      colidx[(b * G + (c0 + t) / M) * 4 + slot] = static_cast<uint8_t>(j);
    }
    __syncthreads();
    // 4. rows x pairs of groups: 2:4 among the 4 kept columns; the tile keeps only the
    //    2 survivors of each group (for the masked output)
    const int pairs = (gpc + 1) / 2;
    const int64_t g_first = c0 / M;                 // even: CW / M is even
    for (int w = t; w < nr * pairs; w += 256) {
      const int r = w / pairs;
      const int pl = w % pairs;
      uint32_t nib[2] = {0x4u, 0x4u};               // a missing last group keeps the padding nibble
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int gl = 2 * pl + h;
        if (gl >= gpc) break;
        uint16_t* a = tile + r * CW + gl * M;
        const uint8_t* o = offs + gl * 4;
        const uint32_t lo = static_cast<uint32_t>(a[o[0]]) | (static_cast<uint32_t>(a[o[1]]) << 16);
        const uint32_t hi = static_cast<uint32_t>(a[o[2]]) | (static_cast<uint32_t>(a[o[3]]) << 16);
        nib[h] = pick2_nibble(lo, hi);
        *reinterpret_cast<uint32_t*>(vals + (r0 + r) * ldv + 2 * (g_first + gl)) = kept_pair(lo, hi, nib[h]);
        if (Am) {
          const int k0 = o[nib[h] & 3u], k1 = o[nib[h] >> 2];
          for (int q = 0; q < M; ++q)
            if (q != k0 && q != k1) a[q] = 0;
        }
      }
      meta[(r0 + r) * ldm + (g_first + 2 * pl) / 2] = static_cast<uint8_t>(nib[0] | (nib[1] << 4));
    }
    if (Am) {
      __syncthreads();
      for (int i = t; i < nchunks; i += 256)
        *reinterpret_cast<uint4*>(Am + (r0 + i / cpr) * ldam + c0 + (i % cpr) * 8) =
            *reinterpret_cast<const uint4*>(tile + (i / cpr) * CW + (i % cpr) * 8);
    }
    __syncthreads();
  }
}

// V:2:M prune for groups of M <= 32 columns: persistent, TMA-fed, two tile buffers,
// warp-specialised so that the serial column sums of one item overlap the prune of
// the previous one.
// Work item = (block of V rows, 64 * CWB columns), loaded as CWB boxes [V][64] with
// the 128B swizzle: the 16-byte chunk c of row r sits at chunk c ^ (r & 7) of its
// 128-byte row, so a warp reading the same columns of 8 rows, or whole rows, meets
// no bank conflict. (CWB = 2 for V <= 128: each serial column pass then covers as
// many bytes as one pass over 256 rows.)
//   norm warps (64 * CWB threads), item k: column norms over the block, rows in
//     order (fp32, sequential: the oracle's order), one column per thread; per group
//     the 4 columns of largest norm (ties: lower column), their slots and byte
//     offsets in a row, and for each 2:4 outcome a table of byte selectors that builds
//     the group's dense masked form from the kept pair; then stage k & 1 is published.
//   unit warps (256 threads), item k - 1 meanwhile: thread -> (row, group), the group
//     fixed for the item and the rows 256 / (groups per row) apart (a multiple of 8,
//     so the swizzle of the thread's rows is fixed too): the 4 kept values are read
//     from shared memory, 2:4 among them gives the packed pair and the metadata nibble
//     (a pair of groups is joined across neighbouring lanes), and the masked group --
//     zeros with the two survivors in place -- is written straight from registers.
//     M = 4 keeps every column: thread -> (row, two groups), one 16-byte chunk.
//   When the unit warps are done with item k, their first thread refills the buffer
//   with item k + 2. Stage k & 1 is rewritten only for item k + 2, whose tile cannot
//   arrive before that point, so the stages need no barrier of their own.
template <int M, int CWB>
__global__ void __launch_bounds__(64 * CWB + 256, 3) vnm_prune_swz_kernel(
    const __grid_constant__ CUtensorMap tmA, int64_t rows, int64_t cols, int V, int sub_bytes, int64_t n_items,
    int64_t nbx, uint8_t* __restrict__ colidx, uint16_t* __restrict__ vals, int64_t ldv,
    uint8_t* __restrict__ meta, int64_t ldm, uint16_t* Am, int64_t ldam, int* status) {
  static_assert(M >= 4 && M <= 32 && (M & (M - 1)) == 0, "groups of 4, 8, 16 or 32 columns");
  static_assert(CWB == 1 || CWB == 2, "one or two 64-column boxes per item");
  constexpr int CW = 64 * CWB;              // columns per item
  constexpr int GR = M == 4 ? 8 : 64 / M;   // thread units per 64-column box row
  constexpr int UR = GR * CWB;              // thread units per item row
  constexpr int RSTEP = 256 / UR;           // rows between a unit thread's units
  constexpr int MW = M / 2;                 // 32-bit words per group
  constexpr int kNormThreads = CW;
  constexpr int kUnitThreads = 256;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(4) uint8_t offs[2][CW];   // [stage][group][slot]: kept column within the group
  __shared__ __align__(4) uint8_t boff[2][CW];   // [stage][group][slot]: its byte offset in a box row, unswizzled
  __shared__ __align__(16) uint16_t mtab[2][M == 4 ? 8 : 512 * CWB];  // [stage][group][nibble][word]
  __shared__ __align__(8) uint64_t full[2];
  __shared__ __align__(8) uint64_t sel_full[2];
  // 1024-byte aligned (the 128B swizzle), offset from the shared-memory pointer itself so
  // that the compiler keeps shared-memory (not generic) loads
  uint8_t* tiles = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int t = threadIdx.x;
  const int64_t G = cols / M;
  const int buf_bytes = CWB * sub_bytes;
  auto load = [&](int64_t it, int q) {
    mbar_arrive_expect_tx(&full[q], static_cast<uint32_t>(CWB * V * 128));
#pragma unroll
    for (int j = 0; j < CWB; ++j)
      tma_load_2d(tiles + q * buf_bytes + j * sub_bytes, &tmA, &full[q], static_cast<int>((it % nbx) * CW + 64 * j),
                  static_cast<int>((it / nbx) * V));
  };
  if (t == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&sel_full[0], 1);
    mbar_init(&sel_full[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (t == 0) {
    load(blockIdx.x, 0);
    if (blockIdx.x + gridDim.x < n_items) load(blockIdx.x + gridDim.x, 1);
  }
  if (t < kNormThreads) {
    // ------------------------------------------------------------ norm warps
    for (int64_t item = blockIdx.x, k = 0; item < n_items; item += gridDim.x, ++k) {
      const int q = static_cast<int>(k & 1);
      if (!p24_wait_for_idle(&full[q], static_cast<uint32_t>(k >> 1) & 1u, P24_WAIT_NS, status)) return;
      const int64_t b = item / nbx;
      const int64_t c0 = (item % nbx) * CW;
      const int nr = static_cast<int>(min(rows - b * V, static_cast<int64_t>(V)));
      const int ncol = static_cast<int>(min(static_cast<int64_t>(CW), cols - c0));  // multiple of 8 and of M
      if (M == 4) {
        // every column is kept (byte stores: the caller's colidx needs no alignment)
        if (t < ncol) colidx[(b * G + c0 / 4) * 4 + t] = static_cast<uint8_t>(t & 3);
      } else {
        const uint8_t* tile = tiles + q * buf_bytes + (t >> 6) * sub_bytes;
        const int cl = t & 63;  // column within its box
        // column norms, one column per thread: 16 rows' loads issued ahead of their
        // sequential additions (|x| is the value with its sign bit cleared)
        uint32_t kt = 0;
        if (t < ncol) {
          const int cb = (cl >> 3) << 4, cw = (cl & 7) * 2;
          float sum = 0.f;
          int r = 0;
          for (; r + 16 <= nr; r += 16) {
            uint32_t x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
              x[j] = *reinterpret_cast<const uint16_t*>(tile + (r + j) * 128 + (cb ^ ((j & 7) << 4)) + cw);
#pragma unroll
            for (int j = 0; j < 16; ++j) sum += fabsf(__uint_as_float(x[j] << 16));
          }
          for (; r < nr; ++r)
            sum += fabsf(__uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(
                                             tile + r * 128 + (cb ^ ((r & 7) << 4)) + cw))
                                         << 16));
          kt = (sum != sum) ? 0x7FC00000u : __float_as_uint(sum);
        }
        // the 4 kept columns of each group (ties: lower column): a group of M <= 32
        // columns lies inside one warp, so the keys come by shuffle and the slots by ballot
        const int lane = t & 31, j = t % M, gl0 = lane - j;
        int beat = 0;
#pragma unroll
        for (int c = 0; c < M; ++c) {
          const uint32_t kc = __shfl_sync(0xFFFFFFFFu, kt, gl0 + c);
          beat += (kc > kt || (kc == kt && c < j)) ? 1 : 0;
        }
        const bool kp = t < ncol && beat < 4;
        const uint32_t km = __ballot_sync(0xFFFFFFFFu, kp);
        const uint32_t gmask = (M == 32 ? 0xFFFFFFFFu : ((1u << M) - 1u)) << gl0;
        if (kp) {
          const int slot = __popc(km & gmask & ((1u << lane) - 1u));
          offs[q][(t / M) * 4 + slot] = static_cast<uint8_t>(j);
          boff[q][(t / M) * 4 + slot] = static_cast<uint8_t>(((cl >> 3) << 4) | ((cl & 7) << 1));
          colidx[(b * G + (c0 + t) / M) * 4 + slot] = static_cast<uint8_t>(j);
        }
        __syncwarp();
        // masked-group selectors: entry (group, nibble), word w takes from the kept pair
        // (v0 in bytes 0-1, v1 in bytes 2-3) whichever survivor sits in column 2w (low
        // half) and 2w + 1 (high half); byte 4 reads the zero operand. The lanes of a
        // group share its 16 entries.
        if (t < ncol) {
          const int g = t / M;
          for (int nb2 = j; nb2 < 16; nb2 += M) {
            const int i0 = nb2 & 3, i1 = nb2 >> 2;
            const int s0 = i0 < i1 ? offs[q][g * 4 + i0] : -1, s1 = i0 < i1 ? offs[q][g * 4 + i1] : -1;
#pragma unroll
            for (int w = 0; w < MW; ++w) {
              const uint32_t lo = (s0 == 2 * w) ? 0x10u : (s1 == 2 * w) ? 0x32u : 0x44u;
              const uint32_t hi = (s0 == 2 * w + 1) ? 0x10u : (s1 == 2 * w + 1) ? 0x32u : 0x44u;
              mtab[q][(g * 16 + nb2) * MW + w] = static_cast<uint16_t>(lo | (hi << 8));
            }
          }
        }
      }
      named_bar_sync(2, kNormThreads);
      if (t == 0) mbar_arrive(&sel_full[q]);
    }
    return;
  }
  // -------------------------------------------------------------- unit warps
  const int tu = t - kNormThreads;
  const int lane = tu & 31;
  const int u = tu % UR, rt = tu / UR;    // this thread's unit and first row
  const int sw = (rt & 7) << 4;           // the swizzle of all its rows
  const int nk = (V + RSTEP - 1) / RSTEP; // units per thread per item (uniform)
  const int ub = (u / GR) * sub_bytes;    // the unit's box within a buffer
  for (int64_t item = blockIdx.x, k = 0; item < n_items; item += gridDim.x, ++k) {
    const int q = static_cast<int>(k & 1);
    const uint32_t par = static_cast<uint32_t>(k >> 1) & 1u;
    if (!p24_wait_for_idle(&sel_full[q], par, P24_WAIT_NS, status)) return;
    if (!p24_wait_for(&full[q], par, P24_WAIT_NS, status)) return;
    const uint8_t* tile = tiles + q * buf_bytes + ub;
    const int64_t b = item / nbx;
    const int64_t c0 = (item % nbx) * CW;
    const int64_t r0 = b * V;
    const int nr = static_cast<int>(min(rows - r0, static_cast<int64_t>(V)));
    const int ncol = static_cast<int>(min(static_cast<int64_t>(CW), cols - c0));
    const int uvalid = M == 4 ? ncol / 8 : ncol / M;
    const int64_t g_first = c0 / M;
    if (M == 4) {
      const uint8_t* p = tile + rt * 128 + (((u % GR) << 4) ^ sw);
      for (int kk = 0; kk < nk; ++kk) {
        const int r = rt + kk * RSTEP;
        if (r < nr && u < uvalid) {
          const uint4 v = *reinterpret_cast<const uint4*>(p + kk * RSTEP * 128);
          const uint32_t n0 = pick2_nibble(v.x, v.y), n1 = pick2_nibble(v.z, v.w);
          *reinterpret_cast<uint2*>(vals + (r0 + r) * ldv + 2 * (g_first + 2 * u)) =
              make_uint2(kept_pair(v.x, v.y, n0), kept_pair(v.z, v.w, n1));
          meta[(r0 + r) * ldm + g_first / 2 + u] = static_cast<uint8_t>(n0 | (n1 << 4));
          if (Am) {
            uint4 m;
            masked_group(v.x, v.y, n0, m.x, m.y);
            masked_group(v.z, v.w, n1, m.z, m.w);
            *reinterpret_cast<uint4*>(Am + (r0 + r) * ldam + c0 + 8 * u) = m;
          }
        }
      }
    } else {
      const uint32_t bo4 = *reinterpret_cast<const uint32_t*>(&boff[q][u * 4]);
      const int a0 = static_cast<int>(bo4 & 0xFFu) ^ sw, a1 = static_cast<int>((bo4 >> 8) & 0xFFu) ^ sw;
      const int a2 = static_cast<int>((bo4 >> 16) & 0xFFu) ^ sw, a3 = static_cast<int>(bo4 >> 24) ^ sw;
      const uint8_t* p = tile + rt * 128;
      const uint16_t* tb = &mtab[q][u * 16 * MW];
      // two rows (RSTEP apart) per iteration: their 8 loads are issued before either is used
      for (int kk = 0; kk < nk; kk += 2) {
        uint32_t v[2][4];
        bool valid[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = rt + (kk + h) * RSTEP;
          valid[h] = kk + h < nk && r < nr && u < uvalid;
          if (valid[h]) {
            const uint8_t* pr = p + (kk + h) * RSTEP * 128;
            v[h][0] = *reinterpret_cast<const uint16_t*>(pr + a0);
            v[h][1] = *reinterpret_cast<const uint16_t*>(pr + a1);
            v[h][2] = *reinterpret_cast<const uint16_t*>(pr + a2);
            v[h][3] = *reinterpret_cast<const uint16_t*>(pr + a3);
          }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = rt + (kk + h) * RSTEP;
          uint32_t nib = 0x4u;  // a missing group keeps the padding nibble
          if (valid[h]) {
            const uint32_t lo = v[h][0] | (v[h][1] << 16), hi = v[h][2] | (v[h][3] << 16);
            nib = pick2_nibble(lo, hi);
            const uint32_t pair = kept_pair(lo, hi, nib);
            *reinterpret_cast<uint32_t*>(vals + (r0 + r) * ldv + 2 * (g_first + u)) = pair;
            if (Am) {
              uint16_t* dst = Am + (r0 + r) * ldam + c0 + u * M;
              const uint16_t* sel = tb + nib * MW;
#pragma unroll
              for (int c = 0; c < M / 8; ++c) {
                const uint2 s01 = *reinterpret_cast<const uint2*>(sel + 4 * c);
                *reinterpret_cast<uint4*>(dst + 8 * c) =
                    make_uint4(__byte_perm(pair, 0u, s01.x & 0xFFFFu), __byte_perm(pair, 0u, s01.x >> 16),
                               __byte_perm(pair, 0u, s01.y & 0xFFFFu), __byte_perm(pair, 0u, s01.y >> 16));
              }
            }
          }
          // groups 2p and 2p+1 are lanes 2p' and 2p'+1 (UR is even, so a lane pair shares a row)
          const uint32_t other = __shfl_down_sync(0xFFFFFFFFu, nib, 1);
          if (valid[h] && (lane & 1) == 0) {
            const uint32_t hi_nib = (u + 1 < uvalid) ? other : 0x4u;
            meta[(r0 + r) * ldm + (g_first + u) / 2] = static_cast<uint8_t>(nib | (hi_nib << 4));
          }
        }
      }
    }
    // every unit thread is done with buffer q: refill it with item k + 2
    named_bar_sync(1, kUnitThreads);
    if (tu == 0 && item + 2 * gridDim.x < n_items) {
      fence_proxy_async_smem();
      load(item + 2 * static_cast<int64_t>(gridDim.x), q);
    }
  }
}

// One launch of vnm_prune_swz_kernel<M, CWB> with as many CTAs per SM as fit.
template <int M, int CWB>
cudaError_t launch_vnm_prune_swz(const CUtensorMap& tm, int64_t rows, int64_t cols, int V, int sub_bytes,
                                 int64_t nb, uint8_t* colidx, const p24_sparse& out, uint16_t* am, int64_t ldam,
                                 int* status, int sms, cudaStream_t s) {
  constexpr int kThreads = 64 * CWB + 256;
  const int smem = 2 * CWB * sub_bytes + 1024;  // + the 1024-byte alignment of the swizzled buffers
  static std::once_flag once[64];
  static cudaError_t attr[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::call_once(once[dev], [&] {
    attr[dev] = cudaFuncSetAttribute(vnm_prune_swz_kernel<M, CWB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     64 * 1024 + 1024);
  });
  if (attr[dev] != cudaSuccess) return attr[dev];
  static thread_local int occ_smem[64], occ_ctas[64];
  if (occ_smem[dev] != smem) {
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, vnm_prune_swz_kernel<M, CWB>, kThreads, smem);
    if (e != cudaSuccess) return e;
    occ_ctas[dev] = std::max(1, n);
    occ_smem[dev] = smem;
  }
  const int64_t nbx = (cols + 64 * CWB - 1) / (64 * CWB);
  const int64_t n_items = nb * nbx;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(n_items, static_cast<int64_t>(sms) * occ_ctas[dev]));
  return launch_pdl(vnm_prune_swz_kernel<M, CWB>, dim3(grid), dim3(kThreads), smem, s, tm, rows, cols, V, sub_bytes,
                    n_items, nbx, colidx, static_cast<uint16_t*>(out.vals), out.ldv, out.meta, out.ldm, am, ldam,
                    status);
}

// The same prune as a persistent kernel: work item = (row block, CW-column chunk);
// each item's V x CW tile is brought into shared memory by one TMA box while the
// previous item is processed (two buffers), so the HBM stream overlaps the serial
// fp32 column sums. Rows past the matrix arrive as zeros and add nothing to a sum.
// After the prune pass has zeroed the dropped entries in shared memory, the tile is
// the dense masked output and is written back with 16-byte stores.
__global__ void __launch_bounds__(256) vnm_compress_tma_kernel(
    const __grid_constant__ CUtensorMap tmA, int64_t rows, int64_t cols, int V, int M, int CW, int64_t n_items,
    int64_t nbx, uint8_t* __restrict__ colidx, uint16_t* __restrict__ vals, int64_t ldv,
    uint8_t* __restrict__ meta, int64_t ldm, uint16_t* Am, int64_t ldam, int* status) {
  extern __shared__ __align__(128) uint16_t tiles[];  // 2 x [V][CW]
  __shared__ uint32_t key[256];
  __shared__ uint8_t kept[256];
  __shared__ uint8_t offs[256];
  __shared__ __align__(8) uint64_t full[2];
  const int t = threadIdx.x;
  const int64_t G = cols / M;
  const int j = t % M, gstart = t - j;
  const int tile_elems = V * CW;
  if (t == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    fence_barrier_init();
  }
  __syncthreads();
  int64_t item = blockIdx.x;
  if (t == 0 && item < n_items) {
    mbar_arrive_expect_tx(&full[0], static_cast<uint32_t>(tile_elems * 2));
    tma_load_2d(tiles, &tmA, &full[0], static_cast<int>((item % nbx) * CW), static_cast<int>((item / nbx) * V));
  }
  for (int i = 0; item < n_items; ++i, item += gridDim.x) {
    const int buf = i & 1;
    const int64_t next = item + gridDim.x;
    if (t == 0 && next < n_items) {
      // the other buffer was last read and written by this CTA's threads (generic
      // proxy) before the barrier that ended the previous item
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(&full[buf ^ 1], static_cast<uint32_t>(tile_elems * 2));
      tma_load_2d(tiles + (buf ^ 1) * tile_elems, &tmA, &full[buf ^ 1], static_cast<int>((next % nbx) * CW),
                  static_cast<int>((next / nbx) * V));
    }
    if (!p24_wait_for(&full[buf], (i >> 1) & 1, P24_WAIT_NS, status)) return;
    uint16_t* tile = tiles + buf * tile_elems;
    const int64_t b = item / nbx;
    const int64_t c0 = (item % nbx) * CW;
    const int64_t r0 = b * V;
    const int nr = static_cast<int>(min(rows - r0, static_cast<int64_t>(V)));
    const int ncol = static_cast<int>(min(static_cast<int64_t>(CW), cols - c0));
    const int gpc = ncol / M;
    // 1. column norm over the block, rows in order
    if (t < ncol) {
      float sum = 0.f;
      for (int r = 0; r < nr; ++r) sum += __uint_as_float(static_cast<uint32_t>(tile[r * CW + t] & 0x7FFFu) << 16);
      key[t] = (sum != sum) ? 0x7FC00000u : __float_as_uint(sum);
    }
    __syncthreads();
    // 2. selection and slot
    if (t < ncol) {
      const uint32_t k = key[t];
      int beat = 0;
      for (int q = 0; q < M; ++q) {
        const uint32_t kq = key[gstart + q];
        beat += (kq > k || (kq == k && q < j)) ? 1 : 0;
      }
      kept[t] = beat < 4 ? 1 : 0;
    }
    __syncthreads();
    if (t < ncol && kept[t]) {
      int slot = 0;
      for (int q = 0; q < j; ++q) slot += kept[gstart + q];
      offs[(t / M) * 4 + slot] = static_cast<uint8_t>(j);
      colidx[(b * G + (c0 + t) / M) * 4 + slot] = static_cast<uint8_t>(j);
    }
    __syncthreads();
    // 3. rows x pairs of groups
    const int pairs = (gpc + 1) / 2;
    const int64_t g_first = c0 / M;
    for (int w = t; w < nr * pairs; w += 256) {
      const int r = w / pairs;
      const int pl = w % pairs;
      uint32_t nib[2] = {0x4u, 0x4u};
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int gl = 2 * pl + h;
        if (gl >= gpc) break;
        uint16_t* a = tile + r * CW + gl * M;
        const uint8_t* o = offs + gl * 4;
        const uint32_t lo = static_cast<uint32_t>(a[o[0]]) | (static_cast<uint32_t>(a[o[1]]) << 16);
        const uint32_t hi = static_cast<uint32_t>(a[o[2]]) | (static_cast<uint32_t>(a[o[3]]) << 16);
        nib[h] = pick2_nibble(lo, hi);
        *reinterpret_cast<uint32_t*>(vals + (r0 + r) * ldv + 2 * (g_first + gl)) = kept_pair(lo, hi, nib[h]);
        if (Am) {
          const int k0 = o[nib[h] & 3u], k1 = o[nib[h] >> 2];
          for (int q = 0; q < M; ++q)
            if (q != k0 && q != k1) a[q] = 0;
        }
      }
      meta[(r0 + r) * ldm + (g_first + 2 * pl) / 2] = static_cast<uint8_t>(nib[0] | (nib[1] << 4));
    }
    if (Am) {
      __syncthreads();
      const int cpr = ncol / 8;
      for (int q = t; q < nr * cpr; q += 256)
        *reinterpret_cast<uint4*>(Am + (r0 + q / cpr) * ldam + c0 + (q % cpr) * 8) =
            *reinterpret_cast<const uint4*>(tile + (q / cpr) * CW + (q % cpr) * 8);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------- double prune
constexpr int kDpRows = 128, kDpCols = 128, kDpChunks = kDpCols / 8;

struct DpArgs {
  const uint16_t* W;        // dense input (kFromDense)
  int64_t ldw;
  const uint16_t* fv_in;    // forward values / metadata: read (compressed input) or written
  uint16_t* fv_out;
  int64_t ldfv;
  const uint8_t* fm_in;
  uint8_t* fm_out;
  int64_t ldfm;
  int64_t rows, cols;
  uint16_t* tv;             // W_bwd^T values / metadata
  int64_t ldtv;
  uint8_t* tm;
  int64_t ldtm;
  uint16_t* Wm;             // optional dense forward-masked copy: [rows, ldwm], or with
  int64_t ldwm;             // kMaskedT its transpose [cols, ldwm]
  uint32_t hi16;            // 2^16 (see pick2_code_mh)
};

// One 128 x 128 tile. kEdge: the tile crosses the last row or column, so every
// access is checked; interior tiles (all but a thin border) skip the checks.
template <bool kFromDense, bool kMasked, bool kEdge, bool kMaskedT>
__device__ __forceinline__ void dp_tile(const DpArgs& p, int64_t row0, int64_t col0, uint4* tile,
                                        const uint2* ptab) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int c = threadIdx.x & (kDpChunks - 1);  // load phase: chunk of the thread
  const int rb = threadIdx.x >> 4;               // load phase: first row of the thread
  const int64_t e = col0 + 8 * c;
  const int64_t r_first = row0 + rb;

  // ---------------- load (+ forward prune)
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t row = r_first + 16 * i;
    v[i] = make_uint4(0, 0, 0, 0);
    const bool full = !kEdge || (row < p.rows && e + 8 <= p.cols);
    const bool half = kEdge && row < p.rows && !full && e + 4 <= p.cols;
    if (kFromDense) {
      if (full) v[i] = ld_stream_v4(p.W + row * p.ldw + e);
      else if (half) {
        const uint2 x = __ldcs(reinterpret_cast<const uint2*>(p.W + row * p.ldw + e));
        v[i].x = x.x;
        v[i].y = x.y;
      }
    } else if (full || half) {
      const uint32_t mb = p.fm_in[row * p.ldfm + e / 8];
      if (full) {
        const uint2 pr = *reinterpret_cast<const uint2*>(p.fv_in + row * p.ldfv + e / 2);
        expand_group(pr.x, mb & 0xFu, v[i].x, v[i].y);
        expand_group(pr.y, mb >> 4, v[i].z, v[i].w);
      } else {
        const uint32_t pr = *reinterpret_cast<const uint32_t*>(p.fv_in + row * p.ldfv + e / 2);
        expand_group(pr, mb & 0xFu, v[i].x, v[i].y);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = rb + 16 * i;
    const int64_t row = row0 + r;
    if (kFromDense) {
      const bool full = !kEdge || (row < p.rows && e + 8 <= p.cols);
      const bool half = kEdge && row < p.rows && !full && e + 4 <= p.cols;
      if (full || half) {
        const uint2 r0 = ptab[pick2_code_mh(v[i].x, v[i].y, p.hi16)];
        const uint32_t n0 = r0.x >> 16;
        const uint32_t k0 = __byte_perm(v[i].x, v[i].y, r0.x);
        v[i].x = __byte_perm(v[i].x, 0u, r0.y);
        v[i].y = __byte_perm(v[i].y, 0u, r0.y >> 16);
        if (full) {
          const uint2 r1 = ptab[pick2_code_mh(v[i].z, v[i].w, p.hi16)];
          const uint32_t n1 = r1.x >> 16;
          const uint32_t k1 = __byte_perm(v[i].z, v[i].w, r1.x);
          v[i].z = __byte_perm(v[i].z, 0u, r1.y);
          v[i].w = __byte_perm(v[i].w, 0u, r1.y >> 16);
          *reinterpret_cast<uint2*>(p.fv_out + row * p.ldfv + e / 2) = make_uint2(k0, k1);
          p.fm_out[row * p.ldfm + e / 8] = static_cast<uint8_t>(n0 | (n1 << 4));
          if (kMasked) *reinterpret_cast<uint4*>(p.Wm + row * p.ldwm + e) = v[i];
        } else {
          *reinterpret_cast<uint32_t*>(p.fv_out + row * p.ldfv + e / 2) = k0;
          p.fm_out[row * p.ldfm + e / 8] = static_cast<uint8_t>(n0 | 0x40u);
          if (kMasked) *reinterpret_cast<uint2*>(p.Wm + row * p.ldwm + e) = make_uint2(v[i].x, v[i].y);
        }
      }
    }
    tile[r * kDpChunks + (c ^ ((r >> 2) & (kDpChunks - 1)))] = v[i];
  }
  __syncthreads();

  // ---------------- column groups: lane = row quad, warp = 2 chunks (16 columns)
  const int h = lane;
  const int64_t nquads = p.rows / 4;
  const int64_t hq = row0 / 4 + h;  // global quad = group index along W_bwd^T rows
  const bool active = !kEdge || hq < nquads;
  // the quad after an even lane's is inside the matrix unless the tile crosses its end
  const bool next_in = !kEdge || hq + 1 < nquads;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int chunk = 2 * warp + cc;
    const int64_t cbase = col0 + 8 * chunk;
    if (kEdge && cbase >= p.cols) break;  // uniform per warp
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = tile[(4 * h + i) * kDpChunks + (chunk ^ (h & (kDpChunks - 1)))];
    const uint32_t w0[4] = {q[0].x, q[0].y, q[0].z, q[0].w};
    const uint32_t w1[4] = {q[1].x, q[1].y, q[1].z, q[1].w};
    const uint32_t w2[4] = {q[2].x, q[2].y, q[2].z, q[2].w};
    const uint32_t w3[4] = {q[3].x, q[3].y, q[3].z, q[3].w};
    uint16_t* tvp = p.tv + cbase * p.ldtv + 2 * hq;
    uint8_t* tmp = p.tm + cbase * p.ldtm + hq / 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (kEdge && cbase + j >= p.cols) break;  // uniform per warp
      const uint32_t sel = (j & 1) ? 0x7632u : 0x5410u;
      const uint32_t lo = __byte_perm(w0[j >> 1], w1[j >> 1], sel);
      const uint32_t hi = __byte_perm(w2[j >> 1], w3[j >> 1], sel);
      const uint32_t entry = ptab[pick2_code_mh(lo, hi, p.hi16)].x;
      const uint32_t nib = entry >> 16;
      const uint32_t pair = __byte_perm(lo, hi, entry);
      const uint32_t nib_next = __shfl_down_sync(0xFFFFFFFFu, nib, 1);
      if (active) {
        *reinterpret_cast<uint32_t*>(tvp + j * p.ldtv) = pair;
        if ((lane & 1) == 0) tmp[j * p.ldtm] = static_cast<uint8_t>(nib | ((next_in ? nib_next : 0x4u) << 4));
        // the forward-masked quad of column j, transposed: 4 consecutive values of a W^T row
        if (kMaskedT) *reinterpret_cast<uint2*>(p.Wm + (cbase + j) * p.ldwm + 4 * hq) = make_uint2(lo, hi);
      }
    }
  }
  __syncthreads();
}

// A CTA owns a 128-row x 128-column tile of W_fwd. Load phase: coalesced 16-byte
// pieces (thread = row piece), the forward prune of dense input happens here and
// the forward outputs are written straight out; the forward-masked tile goes to
// shared memory with its 16-byte chunks XOR-swizzled by the row quad, so that in
// the column phase a warp (lane = row quad) reads 4 rows x 16 bytes per lane
// without bank conflicts. Column phase: each lane prunes the 4-row column groups
// of its quad and lanes write consecutive groups of a W_bwd^T row (coalesced).
// Each 2:4 decision indexes a 16-row table (pick_row) in shared memory that holds
// the kept pair's byte selector, the masking selectors and the nibble.
// kFromDense: input is the dense W; otherwise the compressed forward matrix.
//
// Interior tiles (whole 128 x 128 blocks) run without bounds checks, four CTAs
// per SM; the border tiles of a ragged matrix (the last partial block column, then
// the last partial block row) run checked in a second, small launch.
template <bool kFromDense, bool kMasked, bool kMaskedT>
__global__ void __launch_bounds__(256, 4) double_prune_interior_kernel(const DpArgs p, int64_t rows_full) {
  __shared__ uint4 tile[kDpRows * kDpChunks];
  __shared__ uint2 ptab[16];
  if (threadIdx.x < 16) ptab[threadIdx.x] = pick_row(threadIdx.x);
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t col0 = static_cast<int64_t>(blockIdx.x) * kDpCols;
  for (int64_t row0 = static_cast<int64_t>(blockIdx.y) * kDpRows; row0 < rows_full;
       row0 += static_cast<int64_t>(gridDim.y) * kDpRows)
    dp_tile<kFromDense, kMasked, false, kMaskedT>(p, row0, col0, tile, ptab);
}

template <bool kFromDense, bool kMasked, bool kMaskedT>
__global__ void __launch_bounds__(256, 2) double_prune_border_kernel(const DpArgs p, int64_t n_col_part,
                                                                    int64_t full_bx, int64_t full_by) {
  __shared__ uint4 tile[kDpRows * kDpChunks];
  __shared__ uint2 ptab[16];
  if (threadIdx.x < 16) ptab[threadIdx.x] = pick_row(threadIdx.x);
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  const int64_t t = blockIdx.x;
  const int64_t bx = t < n_col_part ? full_bx : t - n_col_part;
  const int64_t by = t < n_col_part ? t : full_by;
  dp_tile<kFromDense, kMasked, true, kMaskedT>(p, by * kDpRows, bx * kDpCols, tile, ptab);
}

inline unsigned grid_y(int64_t n) { return static_cast<unsigned>(n < 65535 ? (n < 1 ? 1 : n) : 65535); }

template <bool kFromDense, bool kMasked, bool kMaskedT = false>
cudaError_t launch_double_prune(const DpArgs& a, cudaStream_t s) {
  const int64_t full_bx = a.cols / kDpCols, full_by = a.rows / kDpRows;
  const int64_t nby = (a.rows + kDpRows - 1) / kDpRows;
  if (full_bx > 0 && full_by > 0) {
    dim3 grid(static_cast<unsigned>(full_bx), grid_y(full_by));
    const cudaError_t e = launch_plain(double_prune_interior_kernel<kFromDense, kMasked, kMaskedT>, grid, dim3(256), 0,
                                     s, a, full_by * kDpRows);
    if (e != cudaSuccess) return e;
    count_launch();
  }
  const int64_t n_col_part = (a.cols % kDpCols) ? nby : 0;       // last block column, every block row
  const int64_t n_row_part = (a.rows % kDpRows) ? full_bx : 0;   // last block row, full block columns
  if (n_col_part + n_row_part > 0) {
    const cudaError_t e = launch_plain(double_prune_border_kernel<kFromDense, kMasked, kMaskedT>,
                                     dim3(static_cast<unsigned>(n_col_part + n_row_part)), dim3(256), 0, s, a,
                                     n_col_part, full_bx, full_by);
    if (e != cudaSuccess) return e;
    count_launch();
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------- padding
// Zero values past cols/2 and 0x4 nibbles past the last group, up to the strides.
__global__ void pad_kernel(uint16_t* __restrict__ vals, int64_t ldv, uint8_t* __restrict__ meta, int64_t ldm,
                           int64_t rows, int64_t cols) {
  pdl_wait();
  pdl_trigger();
  const int64_t nv = ldv - cols / 2;
  const int64_t groups = cols / 4;
  const int64_t mb0 = (groups + 1) / 2;  // first byte with no data nibble
  const int64_t nm = ldm - mb0;
  const int64_t per_row = nv + nm;
  const int64_t total = rows * per_row;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / per_row, j = i % per_row;
    if (j < nv) vals[r * ldv + cols / 2 + j] = 0;
    else meta[r * ldm + mb0 + (j - nv)] = 0x44;
  }
}

// ---------------------------------------------------------------- column sums
// Column sums G [M, N] -> out [N] in a fixed order. Pass 1: slab s of
// rows_per_slab consecutive rows is summed top to bottom, one thread per 8 columns
// with 16-byte loads (rows start 16-byte aligned: the boundary checks that), 8 rows
// of loads in flight; a ragged last piece of fewer than 8 columns is read per value.
// Pass 2 adds the slab partials of each column in slab order.
__device__ __forceinline__ void add_bf16x8(float* a, const uint4& v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    a[2 * k] += __uint_as_float(w[k] << 16);
    a[2 * k + 1] += __uint_as_float(w[k] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(256) colsum_partial_kernel(const uint16_t* __restrict__ G, int64_t M, int64_t N,
                                                             int64_t ldg, int64_t rows_per_slab,
                                                             float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  const int64_t c0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 8;
  if (c0 >= N) return;
  const int64_t s = blockIdx.y;
  const int64_t r0 = s * rows_per_slab;
  const int64_t r1 = min(M, r0 + rows_per_slab);
  const int nc = static_cast<int>(min(static_cast<int64_t>(8), N - c0));
  float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  const uint16_t* g = G + r0 * ldg + c0;
  if (nc == 8) {
    int64_t r = r0;
    for (; r + 8 <= r1; r += 8, g += 8 * ldg) {
      uint4 v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(g + i * ldg));
#pragma unroll
      for (int i = 0; i < 8; ++i) add_bf16x8(a, v[i]);
    }
    for (; r < r1; ++r, g += ldg) add_bf16x8(a, __ldg(reinterpret_cast<const uint4*>(g)));
  } else {
    for (int64_t r = r0; r < r1; ++r, g += ldg)
      for (int j = 0; j < nc; ++j) a[j] += __uint_as_float(static_cast<uint32_t>(g[j]) << 16);
  }
  float* o = part + s * N + c0;
  for (int j = 0; j < nc; ++j) o[j] = a[j];
}

__global__ void colsum_final_kernel(const float* __restrict__ part, int64_t S, int64_t N, float* __restrict__ out) {
  const int64_t col = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (col >= N) return;
  float a = 0.f;
#pragma unroll 8
  for (int64_t s = 0; s < S; ++s) a += part[s * N + col];
  out[col] = a;
}

// The S partial sums of 32 columns per CTA: warp w adds slabs [w S/8, (w+1) S/8) in
// order, then the 8 warp sums are added in warp order (a fixed order for given S).
__global__ void __launch_bounds__(256) colsum_final_wide_kernel(const float* __restrict__ part, int64_t S,
                                                                int64_t N, float* __restrict__ out) {
  __shared__ float ws[8][32];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t col = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t per = (S + 7) / 8;
  const int64_t s0 = warp * per, s1 = min(S, s0 + per);
  float a = 0.f;
  if (col < N) {
#pragma unroll 8
    for (int64_t sl = s0; sl < s1; ++sl) a += part[sl * N + col];
  }
  ws[warp][lane] = a;
  __syncthreads();
  if (warp == 0 && col < N) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) t += ws[w][lane];
    out[col] = t;
  }
}

// Scratch of p24_colsum_noalloc: a fixed device array, so that the call needs
// no allocation. Every GPU that loads the library holds it until the process
// exits. All calls share it (calls that overlap on the GPU race on it).
__device__ __align__(256) float g_colsum_scratch[kNoAllocColsumScratch];

// Failure-path self test: one thread waits on an mbarrier that nothing ever
// arrives on. The bounded wait expires after limit_ns, records P24_ETIMEOUT in the
// status word and the kernel returns normally (no trap, no hang).
__global__ void selftest_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  p24_wait_for(&bar, 0, limit_ns, status);
}

}  // namespace

// dst [cols, rows] = src [rows, cols]^T for bf16: 32 x 32 tiles through shared
// memory (one padding column against bank conflicts); coalesced on both sides.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ src, int64_t rows,
                                                             int64_t cols, int64_t lds, uint16_t* __restrict__ dst,
                                                             int64_t ldd) {
  __shared__ uint16_t tile[32][33];
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 32, r0 = static_cast<int64_t>(blockIdx.y) * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32 threads
  for (int i = ty; i < 32; i += 8) {
    const int64_t r = r0 + i, c = c0 + tx;
    if (r < rows && c < cols) tile[i][tx] = src[r * lds + c];
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int64_t c = c0 + i, r = r0 + tx;
    if (c < cols && r < rows) dst[c * ldd + r] = tile[tx][i];
  }
}

cudaError_t launch_transpose_bf16(const void* src, int64_t rows, int64_t cols, int64_t lds, void* dst, int64_t ldd,
                                  cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if ((rows + 31) / 32 > 65535) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>((cols + 31) / 32), static_cast<unsigned>((rows + 31) / 32));
  transpose_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(src), rows, cols, lds,
                                              static_cast<uint16_t*>(dst), ldd);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  selftest_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_pad(const p24_sparse& d, cudaStream_t s) {
  const int64_t per_row = (d.ldv - d.cols / 2) + (d.ldm - (d.cols / 4 + 1) / 2);
  if (per_row <= 0 || d.rows == 0) return cudaSuccess;
  const int64_t total = d.rows * per_row;
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 152 * 16);
  const cudaError_t e = launch_pdl(pad_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, s,
                                   static_cast<uint16_t*>(d.vals), d.ldv, d.meta, d.ldm, d.rows, d.cols);
  count_launch();
  return e;
}

cudaError_t launch_compress(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse& out,
                            void* W_masked, int64_t ldwm, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t pieces = (cols + 7) / 8;
  dim3 grid(static_cast<unsigned>((pieces + 1023) / 1024), grid_y(rows));
  const auto* w = static_cast<const uint16_t*>(W);
  auto* v = static_cast<uint16_t*>(out.vals);
  if (W_masked)
    compress_kernel<true><<<grid, 256, 0, s>>>(w, rows, cols, ldw, v, out.ldv, out.meta, out.ldm,
                                               static_cast<uint16_t*>(W_masked), ldwm);
  else
    compress_kernel<false><<<grid, 256, 0, s>>>(w, rows, cols, ldw, v, out.ldv, out.meta, out.ldm, nullptr, 0);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pad(out, s);
}

cudaError_t launch_compress_both(const void* W, int64_t rows, int64_t cols, int64_t ldw, const p24_sparse& fwd,
                                 const p24_sparse& bwdT, void* W_masked, int64_t ldwm, cudaStream_t s,
                                 void* W_masked_T, int64_t ldwmT) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const auto* w = static_cast<const uint16_t*>(W);
  // one dense masked copy at most: row-major (W_masked) or transposed (W_masked_T)
  if (W_masked && W_masked_T) return cudaErrorInvalidValue;
  const DpArgs a{w,       ldw,  nullptr, static_cast<uint16_t*>(fwd.vals), fwd.ldv, nullptr, fwd.meta, fwd.ldm,
                 rows,    cols, static_cast<uint16_t*>(bwdT.vals), bwdT.ldv, bwdT.meta, bwdT.ldm,
                 static_cast<uint16_t*>(W_masked_T ? W_masked_T : W_masked), W_masked_T ? ldwmT : ldwm, 65536u};
  cudaError_t e = W_masked_T ? launch_double_prune<true, false, true>(a, s)
                             : (W_masked ? launch_double_prune<true, true>(a, s) : launch_double_prune<true, false>(a, s));
  if (e != cudaSuccess) return e;
  if ((e = launch_pad(fwd, s)) != cudaSuccess) return e;
  return launch_pad(bwdT, s);
}

cudaError_t launch_vnm_compress(const void* A, int64_t rows, int64_t cols, int64_t lda, int V, int M,
                                uint8_t* colidx, const p24_sparse& out, void* A_masked, int64_t ldam, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t nb = (rows + V - 1) / V;
  if (V <= 256 && cols % 8 == 0 && M <= 32) {
    // groups of at most 32 columns: 64-column swizzled boxes (two per item for V <= 128)
    const int sub_bytes = ((V + 7) / 8) * 1024;
    CUtensorMap tm;
    if (!make_tensor_map_2d(&tm, true, A, cols, rows, lda * 2, 64, V, true)) return cudaErrorInvalidValue;
    int* status = device_status_ptr();
    if (!status) return cudaErrorInvalidDevice;
    static std::once_flag once_w[64];
    static int sms_w[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once_w[dev], [&] {
      int sms = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      sms_w[dev] = sms > 0 ? sms : 1;
    });
    auto* am = static_cast<uint16_t*>(A_masked);
    const bool two = V <= 128;
    switch (M) {
      case 4:
        e = two ? launch_vnm_prune_swz<4, 2>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s)
                : launch_vnm_prune_swz<4, 1>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s);
        break;
      case 8:
        e = two ? launch_vnm_prune_swz<8, 2>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s)
                : launch_vnm_prune_swz<8, 1>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s);
        break;
      case 16:
        e = two ? launch_vnm_prune_swz<16, 2>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s)
                : launch_vnm_prune_swz<16, 1>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s);
        break;
      default:
        e = two ? launch_vnm_prune_swz<32, 2>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s)
                : launch_vnm_prune_swz<32, 1>(tm, rows, cols, V, sub_bytes, nb, colidx, out, am, ldam, status, sms_w[dev], s);
        break;
    }
    count_launch();
    if (e != cudaSuccess) return e;
    return launch_pad(out, s);
  }
  if (V <= 256 && cols % 8 == 0 && 2 * V * (M <= 32 ? 64 : 2 * M) * 2 <= 128 * 1024) {
    // persistent, TMA double-buffered: the narrowest chunk that still holds whole
    // metadata bytes (two groups), two buffers of V x CW
    const int CW = M <= 32 ? 64 : 2 * M;
    const int smem = 2 * V * CW * 2;
    CUtensorMap tm;
    if (!make_tensor_map_2d(&tm, true, A, cols, rows, lda * 2, CW, V)) return cudaErrorInvalidValue;
    int* status = device_status_ptr();
    if (!status) return cudaErrorInvalidDevice;
    static std::once_flag once_t[64];
    static cudaError_t attr_t[64];
    static int per_sm[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once_t[dev], [&] {
      attr_t[dev] = cudaFuncSetAttribute(vnm_compress_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         128 * 1024);
      int sms = 0;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      per_sm[dev] = sms > 0 ? sms : 1;
    });
    if (attr_t[dev] != cudaSuccess) return attr_t[dev];
    const int64_t nbx = (cols + CW - 1) / CW;
    const int64_t n_items = nb * nbx;
    const int64_t ctas_per_sm = std::max<int64_t>(1, std::min<int64_t>(8, (200 * 1024) / (smem + 2048)));
    const int64_t grid = std::min<int64_t>(n_items, per_sm[dev] * ctas_per_sm);
    vnm_compress_tma_kernel<<<static_cast<unsigned>(grid), 256, smem, s>>>(
        tm, rows, cols, V, M, CW, n_items, nbx, colidx, static_cast<uint16_t*>(out.vals), out.ldv, out.meta, out.ldm,
        static_cast<uint16_t*>(A_masked), ldam, status);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pad(out, s);
  }
  if (V <= 256 && cols % 8 == 0) {
    // staged: the block in shared memory (the widest groups, M = 128 with V > 128)
    const int CW = M <= 32 ? 64 : 2 * M;
    const int smem = V * CW * 2;
    static std::once_flag once[64];
    static cudaError_t attr_err[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::call_once(once[dev], [&] {
      attr_err[dev] = cudaFuncSetAttribute(vnm_compress_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           256 * 256 * 2);
    });
    if (attr_err[dev] != cudaSuccess) return attr_err[dev];
    dim3 grid(static_cast<unsigned>((cols + CW - 1) / CW), grid_y(nb));
    vnm_compress_staged_kernel<<<grid, 256, smem, s>>>(
        static_cast<const uint16_t*>(A), rows, cols, lda, V, M, CW, colidx, static_cast<uint16_t*>(out.vals),
        out.ldv, out.meta, out.ldm, static_cast<uint16_t*>(A_masked), ldam);
    count_launch();
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pad(out, s);
  }
  if (A_masked) return cudaErrorInvalidValue;  // the masked output needs the staged kernel (V <= 256)
  dim3 grid(static_cast<unsigned>((cols + kVnmCols - 1) / kVnmCols), grid_y(nb));
  vnm_compress_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(A), rows, cols, lda, V, M, colidx,
                                            static_cast<uint16_t*>(out.vals), out.ldv, out.meta, out.ldm);
  count_launch();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_pad(out, s);
}

cudaError_t launch_transpose_repack(const p24_sparse& fwd, const p24_sparse& bwdT, cudaStream_t s, void* W_masked_T,
                                    int64_t ldwmT) {
  const int64_t rows = fwd.rows, cols = fwd.cols;
  if (rows == 0 || cols == 0) return cudaSuccess;
  const DpArgs a{nullptr, 0,    static_cast<const uint16_t*>(fwd.vals), nullptr, fwd.ldv, fwd.meta, nullptr, fwd.ldm,
                 rows,    cols, static_cast<uint16_t*>(bwdT.vals), bwdT.ldv, bwdT.meta, bwdT.ldm,
                 static_cast<uint16_t*>(W_masked_T), ldwmT, 65536u};
  const cudaError_t e = W_masked_T ? launch_double_prune<false, false, true>(a, s) : launch_double_prune<false, false>(a, s);
  if (e != cudaSuccess) return e;
  return launch_pad(bwdT, s);
}

int64_t colsum_slabs(int64_t M) {
  int64_t S = (M + 127) / 128;
  if (S > 1024) S = 1024;
  if (S < 1) S = 1;
  return S;
}

// Device address of g_colsum_scratch on the current device. Looked up once per
// device (cudaGetSymbolAddress, with that device current) on first use.
float* noalloc_colsum_scratch(cudaError_t* err) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static float* addr[kMaxDevices] = {};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_colsum_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

cudaError_t launch_colsum_noalloc(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (M == 0) return cudaMemsetAsync(out, 0, N * sizeof(float), s);
  cudaError_t err = cudaSuccess;
  float* ws = noalloc_colsum_scratch(&err);
  if (!ws) return err;
  // as many row slabs as the scratch holds partial rows for, at most the usual count
  int64_t S = colsum_slabs(M);
  if (S * N > kNoAllocColsumScratch) S = kNoAllocColsumScratch / N;
  if (S < 1) return cudaErrorInvalidValue;  // rejected on the host before this point
  const int64_t rps = (M + S - 1) / S;
  dim3 grid(static_cast<unsigned>((N + 2047) / 2048), static_cast<unsigned>(S));
  colsum_partial_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(G), M, N, ldg, rps, ws);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colsum_final_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0, s>>>(ws, S, N, out);
  count_launch();
  return cudaGetLastError();
}

// The training step's db_down: as many row slabs as keep about 4 CTAs per SM busy
// (each CTA a slab of at least 16 rows x up to 2048 columns), so that short, wide
// and narrow inputs alike have enough loads in flight; then the parallel final sum.
// (Measured on the 70B dY [16384, 8192]: 8 CTAs per SM 0.063 ms, 4 0.053 ms, 2 0.068 ms.)
int64_t colsum_step_slabs(int64_t M, int64_t N) {
  const int64_t ncb = (N + 2047) / 2048;
  int64_t S = (608 + ncb - 1) / ncb;
  S = std::min<int64_t>(S, (M + 15) / 16);
  S = std::min<int64_t>(S, 1024);
  return std::max<int64_t>(S, 1);
}

cudaError_t launch_colsum_step(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, float* ws,
                               cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (M == 0) return cudaMemsetAsync(out, 0, N * sizeof(float), s);
  const int64_t S = colsum_step_slabs(M, N);
  const int64_t rps = (M + S - 1) / S;
  const int64_t cols_per_cta = std::min<int64_t>(2048, (N + 7) / 8 * 8);
  const int threads = static_cast<int>(((cols_per_cta / 8) + 31) / 32 * 32);
  dim3 grid(static_cast<unsigned>((N + cols_per_cta - 1) / cols_per_cta), static_cast<unsigned>(S));
  cudaError_t e = launch_pdl(colsum_partial_kernel, grid, dim3(threads), 0, s, static_cast<const uint16_t*>(G), M, N,
                             ldg, rps, ws);
  count_launch();
  if (e != cudaSuccess) return e;
  e = launch_pdl(colsum_final_wide_kernel, dim3(static_cast<unsigned>((N + 31) / 32)), dim3(256), 0, s,
                 static_cast<const float*>(ws), S, N, out);
  count_launch();
  return e;
}

cudaError_t launch_colsum(const void* G, int64_t M, int64_t N, int64_t ldg, float* out, float* ws, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (M == 0) return cudaMemsetAsync(out, 0, N * sizeof(float), s);
  const int64_t S = colsum_slabs(M);
  const int64_t rps = (M + S - 1) / S;
  dim3 grid(static_cast<unsigned>((N + 2047) / 2048), static_cast<unsigned>(S));
  colsum_partial_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(G), M, N, ldg, rps, ws);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  colsum_final_kernel<<<static_cast<unsigned>((N + 255) / 256), 256, 0, s>>>(ws, S, N, out);
  count_launch();
  return cudaGetLastError();
}

}  // namespace p24
