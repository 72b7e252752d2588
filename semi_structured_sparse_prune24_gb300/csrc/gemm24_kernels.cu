// gemm24_kernels.cu -- tensor-core GEMMs of the 2:4 FFN training step on
// sm_103a: persistent, warp-specialised kernels with TMA-fed shared-memory
// rings, tcgen05.mma accumulating in tensor memory (TMEM), and fused epilogues.
//
//  spmm_kernel      C[i, j] = sum_r A[i, r] B[j, r], A 2:4-sparse along r
//                   (compressed values in smem, 2-bit metadata in TMEM,
//                   tcgen05.mma.sp), B dense. Used for the forward linear
//                   (A = weight, output written transposed), the double-pruned
//                   backward dX (A = W_bwd^T, SLOPE abstract) and the linear
//                   fed by 2:4 activations (A = activations, straight output).
//  dw_kernel        dW[n, k] = sum_m dY[m, n] X[m, k] kept on the forward 2:4
//                   mask: a dense contraction over tokens (both operands
//                   MN-major), tcgen05.mma kind::f16.
//
// Sources: inno4scale "Success story ESPLAG" ("Research Topic": SpMM on sparse
// tensor cores for the complete training step); SLOPE abstract (double-pruned
// sparse backward); "To 2:4 Sparsity and Beyond" abstract (2:4 weights and
// sparse activations in all FFN matmuls).
//
// Both kernels run as CTA pairs (clusters of 2 CTAs, one per SM) issuing
// cta_group::2 MMAs of M = 256: the two CTAs own adjacent 128-row halves of the A
// tile and each stages half of the shared B tile, which the tensor cores of the
// pair read from both CTAs' shared memory, so B crosses L2 once per pair. The
// leader CTA issues the MMAs; one MMA commit, signalled to both CTAs, frees a
// stage in both. Every load is a plain (non-multicast) TMA copy into the
// issuing CTA's own shared memory.
//
// Roles (warp index): 0 TMA producer, 1 MMA issuer + TMEM owner, 2-5 epilogue
// (warp w reads TMEM lanes 32*(w%4)..+31), 6-9 (spmm only) metadata movers:
// smem -> registers -> TMEM, replacing rows past the matrix with a legal pattern.
//
// TMEM layout of the sparse metadata read by one tcgen05.mma.sp (kind::f16,
// M = 128, K = 32): one 32-bit column over the 128 lanes, rows interleaved in
// blocks of 16. Lane 16b + 8h + i holds, for K-half h (groups 4h..4h+3, 16 bits,
// group 4h in the low nibble), row 16b + i in bits 0-15 and row 16b + 8 + i in
// bits 16-31. (Measured on sm_103a with an identity B operand, which makes the
// accumulator equal to the A operand as the tensor core expanded it.)
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cstdio>
#include <mutex>

#include "p24_internal.h"
#include "p24_ptx.cuh"

namespace p24 {
namespace {

constexpr int kBM = 128;  // MMA M: rows of A per tile = TMEM lanes

// ---------------------------------------------------------------- params
struct SpmmParams {
  int rowsA, rowsB, K;  // K = logical (dense) reduction length
  int tilesA, tilesB, num_tiles, group, nkb;
  __nv_bfloat16* out;
  int64_t ldo;
  const float* bias;
  int relu;
  const uint16_t* gate;
  int64_t ldg;
  float* dbias;              // += column sums (over B rows) of the stored output, per A row
  uint16_t* a24_vals;
  int64_t a24_ldv;
  uint8_t* a24_meta;
  int64_t a24_ldm;
  int* status;
  int b3d;  // B map is 3-D: {64 K, rows, K / 64}; one load brings both 64-K halves of a stage
  int nad;  // dense stages per tile after the sparse ones: A_l [rowsA, r] . B_l [rowsB, r]^T, 64 of r each
  int stall_stage;  // test only: if > 0, both CTAs of cluster 0 skip the loads of their stage number stall_stage - 1
  // V:2:M sparse A (gathered B): A holds, per row block of vnm_V rows and group of vnm_group
  // columns of the logical K, the values at 4 selected columns (condensed, 2:4 along them);
  // vnm_cix [blocks, vnm_G] packs each group's 4 column offsets in one word (byte j =
  // offset j). B is K-outer [vnm_K rows, rowsB columns]; stage rows are gathered by TMA.
  const uint32_t* vnm_cix;
  int vnm_group, vnm_V, vnm_G, vnm_K;
  const uint16_t* vnm_B;  // B [vnm_K, vnm_ldb] (the rows the gather warps copy)
  int64_t vnm_ldb;
};

struct DwParams {
  int N, K, M;  // dW is [N, K]; reduction over M
  int tilesA, tilesB, num_tiles, group, nkb;
  __nv_bfloat16* out;
  int64_t ldo;
  const uint8_t* meta;
  int64_t ldm;
  int* status;
  // Extra tiles past the main ones, unmasked into out2: A-tile pairs >= tilesA_main read a
  // second A operand (out2 rows 0..N2-1), B tiles >= tilesB_main a second B operand
  // (out2 columns 0..K2-1). They share operand panels with the main tiles through L2.
  int tilesA_main, tilesB_main, N2, K2;
  __nv_bfloat16* out2;
  int64_t ldo2;
};

// Grouped raster: consecutive tiles walk `group` A-tiles before the next
// B-tile, so a wave of CTAs shares a few A and B tiles through L2.
__device__ __forceinline__ void tile_coords(int t, int tilesA, int tilesB, int group, int& ta, int& tb) {
  const int per_group = group * tilesB;
  const int g = t / per_group;
  const int first = g * group;
  const int gsize = min(group, tilesA - first);
  const int r = t - g * per_group;
  ta = first + r % gsize;
  tb = r / gsize;
}

// Per 16-bit half: the top bit set where the bf16 value is > 0 (sign clear, magnitude
// nonzero; the sum of a magnitude and 0x7FFF reaches bit 15 exactly when it is nonzero,
// and never carries into the other half).
__device__ __forceinline__ uint32_t bf16_pos_bits(uint32_t w) {
  return (((w & 0x7FFF7FFFu) + 0x7FFF7FFFu) & ~w) & 0x80008000u;
}

// Byte permute with the sign-replicate selector bit (bit 3 of a selector nibble makes
// the result byte the selected byte's top bit, repeated).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
// One byte of gate bits (bit i: value i of a 16-byte piece of 8 bf16) applied to the
// piece. Multiplying a nibble by 2^7 + 2^14 + 2^21 + 2^28 moves its bit k to bit 8k + 7
// (the other partial products land elsewhere and never carry), so each bit becomes a
// byte's top bit; a sign-replicating permute widens two of those bytes into the 16-bit
// masks of one word.
__device__ __forceinline__ void apply_gate(uint4& x, uint32_t byte) {
  const uint32_t s0 = ((byte & 0xFu) * 0x10204080u) & 0x80808080u;
  const uint32_t s1 = ((byte >> 4) * 0x10204080u) & 0x80808080u;
  x.x &= prmt(s0, 0u, 0x9988u);
  x.y &= prmt(s0, 0u, 0xBBAAu);
  x.z &= prmt(s1, 0u, 0x9988u);
  x.w &= prmt(s1, 0u, 0xBBAAu);
}
// Bit i set where bf16 value i of the piece is > 0: the 8 flags sit at bits 15 and 31 of
// the four words; shifts by 15, 13, 11 and 9 put them at bits 0, 2, 4, 6 and 16, 18, 20,
// 22, and folding the upper half down by 15 interleaves them.
__device__ __forceinline__ uint32_t positive_bits(const uint4& x) {
  const uint32_t s = (bf16_pos_bits(x.x) >> 15) | (bf16_pos_bits(x.y) >> 13) | (bf16_pos_bits(x.z) >> 11) |
                     (bf16_pos_bits(x.w) >> 9);
  return (s | (s >> 15)) & 0xFFu;
}

// 2:4 pick on a group held as two words (see prune24_kernels.cu for the key).
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
__device__ __forceinline__ uint32_t kept_pair(uint32_t lo, uint32_t hi, uint32_t nib) {
  const uint32_t i0 = nib & 3u, i1 = nib >> 2;
  return __byte_perm(lo, hi, 0x1010u + i0 * 0x22u + i1 * 0x2200u);
}
__device__ __forceinline__ void mask_group(uint32_t& lo, uint32_t& hi, uint32_t nib) {
  const uint32_t kb = (1u << (nib & 3u)) | (1u << (nib >> 2));
  lo &= ((kb & 1u) ? 0x0000FFFFu : 0u) | ((kb & 2u) ? 0xFFFF0000u : 0u);
  hi &= ((kb & 4u) ? 0x0000FFFFu : 0u) | ((kb & 8u) ? 0xFFFF0000u : 0u);
}

__device__ __forceinline__ void tc_st_32x32b_x1(uint32_t taddr, uint32_t a) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(a) : "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 16 consecutive 32-bit columns of the warp's 32 lanes <- / -> 16 registers per thread.
__device__ __forceinline__ void tc_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tc_ld_32x32b_x16_wait(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                 "+r"(r[15])
               :
               : "memory");
}

// ---------------------------------------------------------------- sparse GEMM (CTA pair)
// A cluster of 2 CTAs computes each 256 x BN output tile with pair MMAs
// (tcgen05.mma.sp.cta_group::2, M = 256). CTA c of the pair holds A rows
// 128c..128c+127 of the tile and B rows c*BN/2..(c+1)*BN/2-1, so each SM stages
// and reads only half of B; CTA 0 (the leader) issues the MMAs. Each CTA's TMEM
// holds the accumulator rows and the metadata of its own 128 A rows, in the
// single-CTA layout. The A and B loads of both CTAs complete on the leader's
// `full` barrier; each CTA's metadata tile completes on its own `efull` barrier.
// Per stage (128 logical K, 4 MMAs) per CTA: A 128 x 64 compressed bf16 (128 B
// rows, 128B swizzle), B two boxes of BN/2 x 64 bf16 (128 B rows, 128B swizzle,
// K 0-63 and 64-127). Metadata comes in blocks of 4 stages (512 logical K):
// 128 rows x 64 B (one 32-bit word per MMA per row), in a ring of its own, so
// that a TMA row request carries 64 bytes instead of 16.
constexpr int kEStages = 4;  // stages per metadata block
constexpr int kEBufs = 2;    // metadata ring depth
template <int BN, int STAGES>
struct SpmmSmem {
  static constexpr int kA = kBM * 128;  // bytes per stage
  static constexpr int kBHalf = (BN / 2) * 128;  // one 64-K box of this CTA's B rows
  static constexpr int kB = 2 * kBHalf;
  static constexpr int kE = kBM * 16 * kEStages;  // bytes per metadata block
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kA;
  static constexpr int kOffE = kOffB + STAGES * kB;
  static constexpr int kOffStage = kOffE + kEBufs * kE;  // epilogue transpose, 4 warps x 32x32 bf16
  static constexpr int kOffGate = kOffStage + 4 * 32 * 32 * 2;  // gate words: 4 warps x BN tokens x 32 features
  static constexpr int kOffBar = kOffGate + 4 * BN * 4;
  static constexpr int kBytes = kOffBar + 8 * (4 * STAGES + 2 * kEBufs + 5) + 16;
  static constexpr int kTxPair = 2 * (kA + kB);  // both CTAs' A and B, counted on the leader's barrier
  static constexpr int kTxDense = 2 * (kA + kBHalf);  // a dense stage: A_l 128 x 64, B_l BN/2 x 64 per CTA
};

// TMEM column of the metadata of MMA j (0-3) of stage s: 8-column slots in the
// gaps after the two accumulator buffers ([BN, 256) and [256 + BN, 512)).
template <int BN>
__device__ __forceinline__ uint32_t meta_col(int s, int j) {
  const int k = 4 * s + j;
  if constexpr (BN > 192) return 256 + 8 * k;  // one accumulator buffer: slots fill [256, 256 + 32 STAGES)
  constexpr int kGap = (256 - BN) / 8;  // slots per gap
  return k < kGap ? BN + 8 * k : 256 + BN + 8 * (k - kGap);
}

// ---- pair (cta_group::2) forms
__device__ __forceinline__ uint32_t leader_addr(const void* p) {  // same smem offset in cluster rank 0
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(r) : "r"(smem_u32(p)));
  return r;
}
// Arrive on a barrier of another CTA of the cluster. Default (CTA-scope release)
// semantics: what the arrival publishes is TMEM state already completed by
// tcgen05.wait::st / wait::ld and ordered by tcgen05 fences, so the costly
// cluster-scope release of all prior memory operations is not needed.
__device__ __forceinline__ void arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x, int y,
                                                 int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, "
      "%4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// ---- gathered B (V:2:M): 16-byte copies by threads, tracked on an mbarrier
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once all of this thread's earlier cp.async copies have landed (the
// barrier's count includes this arrival).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_cta() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_mma_sp_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t e_tmem,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.sp.cta_group::2.kind::f16 [%0], %1, %2, [%3], %4, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(e_tmem), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void tc_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}

// Epilogue kinds, fixed at compile time so that the store loops carry no branches
// for features a call does not use.
enum SpmmEpi : int {
  kEpiStore = 0,  // bias and ReLU only
  kEpiFull = 1,   // any of: ReLU' gate, 2:4 activation prune, column sums (transposed output)
};

// Threads that gather B rows in the V:2:M mode (a multiple of 64, at most 512; measured
// on the 70B down GEMM: 128 -> 256 -> 512 threads gave 2.26 -> 2.06 -> 1.93 ms at M = 16384).
#ifndef P24_GATHER_THREADS
#define P24_GATHER_THREADS 512
#endif
constexpr int kGatherThreads = P24_GATHER_THREADS;
static_assert(kGatherThreads % 64 == 0 && kGatherThreads <= 512, "gather threads");

template <int BN, int STAGES, bool kTransOut, int kEpi, bool kGather = false, bool kDrainOk = true>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kGather ? 320 + kGatherThreads : 320, 1)
    spmm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmE, const __grid_constant__ CUtensorMap tmL,
                const __grid_constant__ CUtensorMap tmT, const SpmmParams p) {
  using L = SpmmSmem<BN, STAGES>;
  constexpr int kAccCols = 256;  // accumulator buffer b starts at column 256 * b
  // BN <= 192: two accumulator buffers (the epilogue of a tile overlaps the next
  // tile's main loop), metadata slots in the two gaps; BN > 192: one buffer.
  constexpr int kAccBufs = BN > 192 ? 1 : 2;
  static_assert(BN <= 256 && BN % 16 == 0, "tile width");
  static_assert(kAccBufs == 1 ? 256 + 8 * 4 * STAGES <= 512 : 4 * STAGES <= 2 * ((256 - BN) / 8), "TMEM budget");
  // One accumulator, transposed output: the epilogue drains the tile into bf16 pairs in
  // the columns after the metadata slots, releases the accumulator, then stores from
  // there (unless kDrainOk is false; see the epilogue).
  constexpr bool kDrain = kTransOut && kAccBufs == 1 && kDrainOk;
  constexpr uint32_t kPackCol = 256 + 8 * 4 * STAGES;
  static_assert(!kDrain || kPackCol + BN / 2 <= 512, "TMEM budget of the drained tile");
  // gathered B is staged MN-major: [K rows][N columns] in 64-column, 128B-swizzled atoms
  constexpr uint32_t kIdesc = idesc_bf16(2 * kBM, BN, /*sparse=*/true, false, /*b_mn=*/kGather);
  static_assert(!kGather || (!kTransOut && BN == 256), "gathered B: straight output, N = 256 tiles");
  constexpr uint32_t kIdescDense = idesc_bf16(2 * kBM, BN, /*sparse=*/false, false, false);
  const int nstages = p.nkb + p.nad;  // per tile: sparse stages, then dense ones

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // keeps shared (not generic) accesses
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // leader's is used
  uint64_t* empty = full + STAGES;                                    // leader's commit, both CTAs
  uint64_t* meta_ready = empty + STAGES;                              // leader's is used (8 arrivals)
  uint64_t* efull = meta_ready + STAGES;                              // [kEBufs] own metadata block landed
  uint64_t* eempty = efull + kEBufs;                                  // [kEBufs] own movers done with it
  uint64_t* acc_full = eempty + kEBufs;                               // [2] leader's commit, both CTAs
  uint64_t* acc_empty = acc_full + 2;                                 // [2] leader's is used (8 arrivals)
  uint64_t* spare = acc_empty + 2;
  uint64_t* bfull = spare + 1;                                        // [STAGES] gathered B: own copies landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bfull + STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // gathered B: the leader's `full` also takes the peer's relay arrival
      mbar_init(&full[s], kGather ? 2 : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&meta_ready[s], 8);  // 4 mover warps x 2 CTAs
      if (kGather) mbar_init(&bfull[s], kGatherThreads);  // one arrival per gather thread
    }
    for (int e = 0; e < kEBufs; ++e) {
      mbar_init(&efull[e], 1);
      mbar_init(&eempty[e], 4);      // this CTA's 4 mover warps
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);   // 4 epilogue warps x 2 CTAs
    }
    mbar_init(spare, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmE);
    if (p.nad) {
      tma_prefetch_desc(&tmL);
      tma_prefetch_desc(&tmT);
    }
  }
  if (warp == 1) {  // pair allocation: one warp of each CTA, same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  pdl_wait();  // the previous kernel's outputs (under programmatic launch)
  pdl_trigger();

  if (kGather && warp >= 10) {
    // ------------------------------------------------ gather warps (both CTAs, gathered B)
    // Stage rows (128 condensed K = 32 groups of 4 selected rows of M) are copied as 16
    // pieces of 16 bytes (this CTA's 128 columns): thread th takes piece c = th % 16 of
    // rows r = RS i + th / 16 (RS = gather threads / 16, i < 128 / RS), so a half warp
    // reads one row's 256 bytes. Row r is row (32 kb + r / 4) M + colidx byte r % 4 of B;
    // its piece c lands in atom c / 8, chunk (c % 8) ^ (r % 8) of the 128B-swizzled
    // MN-major layout. Each thread then arrives once on bfull[s] when its copies have landed.
    constexpr int RS = kGatherThreads / 16;  // rows between a thread's rows
    constexpr int NR = 128 / RS;             // rows per thread per stage
    const int th = threadIdx.x - 320;
    const int c = th & 15;
    const uint32_t sh = 8u * static_cast<uint32_t>((th >> 4) & 3);  // colidx byte of this thread's rows
    const int gofs = th >> 6;                                       // its first row's group
    uint32_t it = 0;
    bool ok = true;
    for (int t = cid; t < p.num_tiles && ok; t += ncl) {
      int ta, tb;
      tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
      const uint32_t* cix = p.vnm_cix + static_cast<int64_t>((ta * 2 * kBM) / p.vnm_V) * p.vnm_G + gofs;
      const uint16_t* bsrc = p.vnm_B + tb * BN + rank * (BN / 2) + 8 * c;
      const uint32_t dst0 = smem_u32(smem + L::kOffB) + (c >> 3) * 16384u;
      uint32_t cw[NR];  // colidx words of this thread's rows for the current stage
#pragma unroll
      for (int i = 0; i < NR; ++i) cw[i] = __ldg(cix + (RS / 4) * i);
      for (int kb = 0; kb < p.nkb; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
        const uint32_t dst = dst0 + static_cast<uint32_t>(s * L::kB);
        const int gb = kb * 32 + gofs;  // every stage is full: the host requires 128 | condensed K
#pragma unroll
        for (int i = 0; i < NR; ++i) {
          const int r = RS * i + (th >> 4);
          const int y = (gb + (RS / 4) * i) * p.vnm_group + static_cast<int>((cw[i] >> sh) & 0xFFu);
          cp_async_16(dst + static_cast<uint32_t>(r) * 128u + ((static_cast<uint32_t>(c & 7) ^ static_cast<uint32_t>(r & 7)) << 4),
                      bsrc + static_cast<int64_t>(y) * p.vnm_ldb);
        }
        cp_async_arrive(&bfull[s]);
        if (kb + 1 < p.nkb) {  // the next stage's words, loaded while this stage's copies fly
#pragma unroll
          for (int i = 0; i < NR; ++i) cw[i] = __ldg(cix + (kb + 1) * 32 + (RS / 4) * i);
        }
      }
    }
    cp_async_wait_all();  // this thread's copies land before the CTA may exit
  } else if (warp == 1 && kGather && !leader) {
    // ------------------------------------------------ relay (second CTA of a gathering pair)
    // This CTA's gathered B for stage s is complete (its own bfull barrier) and lies in
    // its own shared memory: order it for the tensor cores (async proxy) and tell the
    // leader, whose MMAs read it, with a plain remote arrive -- the same hand-over as the
    // metadata movers' TMEM words. (A cluster-scope release here cost 10-12% of the GEMM.)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % STAGES;
          if (!p24_wait(&bfull[s], (it / STAGES) & 1, abort_flag, p.status)) { ok = false; break; }
          fence_proxy_async_cta();
          arrive_cluster(leader_addr(&full[s]));
        }
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0, eit = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int ta, tb;
        tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
        ta = 2 * ta + rank;
        for (int kb = 0; kb < nstages; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (p.stall_stage > 0 && cid == 0 && it + 1 == static_cast<uint32_t>(p.stall_stage)) {
            // test only: no expect_tx and no loads for this stage in either CTA of the
            // pair, so its `full` barrier never completes and the bounded waits expire
            if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
            continue;
          }
          if (kb >= p.nkb) {  // dense stage: 64 of the rank of A_l [rowsA, r] and B_l [rowsB, r]
            if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (leader) mbar_arrive_expect_tx(&full[s], L::kTxDense);
            const uint32_t fullL = leader_addr(&full[s]);
            const int j0 = (kb - p.nkb) * 64;
            tma_load_2d_pair(smem + L::kOffA + s * L::kA, &tmL, fullL, j0, ta * kBM);
            tma_load_2d_pair(smem + L::kOffB + s * L::kB, &tmT, fullL, j0, tb * BN + rank * (BN / 2));
            continue;
          }
          if (kb % kEStages == 0) {  // next metadata block
            const int e = eit % kEBufs;
            if (!p24_wait(&eempty[e], ((eit / kEBufs) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(&efull[e], L::kE);
            tma_load_2d(smem + L::kOffE + e * L::kE, &tmE, &efull[e], (kb / kEStages) * 64, ta * kBM);
            ++eit;
          }
          if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[s], kGather ? 2 * L::kA : L::kTxPair);
          const uint32_t fullL = leader_addr(&full[s]);
          tma_load_2d_pair(smem + L::kOffA + s * L::kA, &tmA, fullL, kb * 64, ta * kBM);
          if (kGather) {
            // B comes from the gather warps
          } else if (p.b3d) {
            tma_load_3d_pair(smem + L::kOffB + s * L::kB, &tmB, fullL, 0, tb * BN + rank * (BN / 2), kb * 2);
          } else {
            tma_load_2d_pair(smem + L::kOffB + s * L::kB, &tmB, fullL, kb * 128, tb * BN + rank * (BN / 2));
            tma_load_2d_pair(smem + L::kOffB + s * L::kB + L::kBHalf, &tmB, fullL, kb * 128 + 64,
                             tb * BN + rank * (BN / 2));
          }
        }
      }
      // Drain: the last issued loads must land before the CTA may exit.
      const uint32_t n_drain = it < STAGES ? it : STAGES;
      for (uint32_t i = 0; i < n_drain; ++i) {
        const uint32_t j = it - 1 - i;
        if (leader) p24_wait_quiet(&full[j % STAGES], (j / STAGES) & 1);
      }
      const uint32_t e_drain = eit < kEBufs ? eit : kEBufs;
      for (uint32_t i = 0; i < e_drain; ++i) {
        const uint32_t j = eit - 1 - i;
        p24_wait_quiet(&efull[j % kEBufs], (j / kEBufs) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader CTA only)
    if (leader) {
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++tl) {
        const int b = kAccBufs == 2 ? (tl & 1) : 0;
        const uint32_t aph = kAccBufs == 2 ? ((tl >> 1) & 1) : (tl & 1);
        if (!p24_wait(&acc_empty[b], aph ^ 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * kAccCols;
        for (int kb = 0; kb < nstages; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (kGather) {
            // A (TMA) and the peer's gathered B (relayed) on `full`, this CTA's gathered B
            // on `bfull`; then order the copies for the tensor cores
            if (!p24_wait(&full[s], ph, abort_flag, p.status) ||
                !p24_wait(&bfull[s], ph, abort_flag, p.status) ||
                !p24_wait(&meta_ready[s], ph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            fence_proxy_async_cta();
          } else if (!p24_wait(&full[s], ph, abort_flag, p.status) ||
                     !p24_wait(&meta_ready[s], ph, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_u32(smem + L::kOffA + s * L::kA);
            const uint32_t b_base = smem_u32(smem + L::kOffB + s * L::kB);
            if (kb < p.nkb) {
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint64_t adesc = smem_desc(a_base + j * 32, 16, 1024, kSwizzle128B);
                // K-major B: 64-K halves of BN/2 rows; gathered (MN-major) B: 32 K rows per
                // MMA in 64-column atoms of 128 rows (atom stride 16 KB, 8-row groups 1 KB)
                const uint64_t bdesc =
                    kGather ? smem_desc(b_base + j * 4096, 16384, 1024, kSwizzle128B)
                            : smem_desc(b_base + (j >> 1) * L::kBHalf + (j & 1) * 64, 16, 1024, kSwizzle128B);
                tc_mma_sp_pair(d_tmem, adesc, bdesc, tmem + meta_col<BN>(s, j), kIdesc, (kb | j) != 0);
              }
            } else {  // dense stage: 4 x K=16 of the low-rank product, into the same accumulator
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint64_t adesc = smem_desc(a_base + j * 32, 16, 1024, kSwizzle128B);
                const uint64_t bdesc = smem_desc(b_base + j * 32, 16, 1024, kSwizzle128B);
                tc_mma_pair(d_tmem, adesc, bdesc, kIdescDense, (kb | j) != 0);
              }
            }
            tc_commit_pair(&empty[s], 0x3);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair(&acc_full[b], 0x3);
        __syncwarp();
      }
      // Make sure no MMA is still running before TMEM is released.
      if (lane == 0) {
        tc_commit_pair(spare, 0x1);
        p24_wait_quiet(spare, 0);
      }
      __syncwarp();
    }
  } else if (warp >= 6 && warp < 10) {
    // ------------------------------------------------ metadata movers (both CTAs)
    // Lane l of quarter q fills TMEM lane 32q + l: rows rA = 32q + (l & 16) + (l & 7)
    // and rA + 8, K-half h = (l >> 3) & 1 of each MMA's 32 metadata bits.
    const int q = warp & 3;
    const int rowA = q * 32 + (lane & 16) + (lane & 7);
    const int rowB = rowA + 8;
    const int h = (lane >> 3) & 1;
    uint32_t it = 0, eit = 0;
    bool ok = true;
    for (int t = cid; t < p.num_tiles && ok; t += ncl) {
      int ta, tb;
      tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
      ta = 2 * ta + rank;
      const bool okA = ta * kBM + rowA < p.rowsA;
      const bool okB = ta * kBM + rowB < p.rowsA;
      for (int kb = 0; kb < nstages; ++kb, ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (it / STAGES) & 1;
        if (kb >= p.nkb) {
          // dense stage: no metadata; arrive once the slot is free, which keeps this
          // barrier's phases in step with the stage ring
          if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          __syncwarp();
          if (lane == 0) arrive_cluster(leader_addr(&meta_ready[s]));
          continue;
        }
        const int eb_i = eit % kEBufs;
        if (kb % kEStages == 0 &&
            !p24_wait(&efull[eb_i], (eit / kEBufs) & 1, abort_flag, p.status)) { ok = false; break; }
        // the stage's TMEM metadata slots are free once the MMAs of their previous use completed
        if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
        const uint8_t* e = smem + L::kOffE + eb_i * L::kE + (kb % kEStages) * 16;
        const uint4 ea = *reinterpret_cast<const uint4*>(e + rowA * 64);
        const uint4 eb = *reinterpret_cast<const uint4*>(e + rowB * 64);
        const uint32_t wa[4] = {ea.x, ea.y, ea.z, ea.w}, wb[4] = {eb.x, eb.y, eb.z, eb.w};
        const uint32_t sh = 16u * h;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a = okA ? (wa[j] >> sh) & 0xFFFFu : 0x4444u;
          const uint32_t b = okB ? (wb[j] >> sh) & 0xFFFFu : 0x4444u;
          tc_st_32x32b_x1(tmem + lane_base + meta_col<BN>(s, j), a | (b << 16));
        }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_cluster(leader_addr(&meta_ready[s]));
        if (kb % kEStages == kEStages - 1 || kb == p.nkb - 1) {  // done with this metadata block
          if (lane == 0) mbar_arrive(&eempty[eb_i]);
          ++eit;
        }
      }
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5, both CTAs)
    const int q = warp & 3;
    uint16_t* stage = reinterpret_cast<uint16_t*>(smem + L::kOffStage) + q * 32 * 32;
    // ReLU' gate of this warp's 32 features: one 32-bit word per token of the tile
    uint32_t* gstage = reinterpret_cast<uint32_t*>(smem + L::kOffGate) + q * BN;
    uint32_t tl = 0;
    for (int t = cid; t < p.num_tiles; t += ncl, ++tl) {
      int ta, tb;
      tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
      ta = 2 * ta + rank;
      const int b = kAccBufs == 2 ? (tl & 1) : 0;
      const uint32_t aph = kAccBufs == 2 ? ((tl >> 1) & 1) : (tl & 1);
      // Transposed output: in the store phase lane l handles tokens 2i, 2i + 1 (i = 8r +
      // l / 4) of each chunk and features n_piece .. n_piece + 7 of the tile.
      const int n_warp = ta * kBM + q * 32;
      const int n_piece = n_warp + (lane & 3) * 8;
      if (kTransOut && kEpi == kEpiFull && p.gate) {
        // The ReLU' gate of this warp's 32 features, one word per token (bit l:
        // gate(m, n_warp + l) > 0), read from the bf16 gate while the tile's main
        // loop still runs, so that no load sits in the epilogue's critical path. Lanes
        // 4i .. 4i + 3 read the 64 contiguous bytes of one token's 32 features, 16 bytes
        // each, so a load instruction covers 8 tokens in whole sectors; 16 loads per lane
        // are issued before any is used, and each lane writes its byte of the word.
        uint8_t* gbytes = reinterpret_cast<uint8_t*>(gstage);
        const int kp = lane & 3;
        const bool col_in = n_warp + 8 * kp < p.rowsA;
        const uint16_t* gcol = p.gate + n_warp + 8 * kp;
        for (int j0 = lane >> 2; j0 < BN; j0 += 128) {
          uint4 x[16];
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int j = j0 + 8 * u;
            const int m = tb * BN + j;
            x[u] = (j < BN && m < p.rowsB && col_in)
                       ? __ldg(reinterpret_cast<const uint4*>(gcol + static_cast<int64_t>(m) * p.ldg))
                       : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const int j = j0 + 8 * u;
            if (j < BN) gbytes[4 * j + kp] = static_cast<uint8_t>(positive_bits(x[u]));
          }
        }
        __syncwarp();
      }
      float dsum[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) dsum[i] = 0.f;
      if (!p24_wait(&acc_full[b], aph, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t acc = tmem + b * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      const int a_row = ta * kBM + q * 32 + lane;  // row of A held by this thread
      if (kTransOut) {
        // out[j, a_row]: token j (B row) x feature a_row (A row). Each chunk of 32 tokens
        // goes through shared memory as bf16 pairs: row i holds tokens 2i and 2i + 1 of
        // the chunk, word f the pair of feature f, at word f ^ 4 (i & 7) (conflict-free
        // both ways). The store phase gives lane l the features n_piece .. n_piece + 7 of
        // token pairs i = 8r + l / 4.
        const float bias_v = (p.bias && a_row < p.rowsA) ? p.bias[a_row] : 0.f;
        auto act_pair = [&](uint32_t a0, uint32_t a1) {
          float f0 = __uint_as_float(a0) + bias_v, f1 = __uint_as_float(a1) + bias_v;
          if (p.relu) {
            f0 = fmaxf(f0, 0.f);
            f1 = fmaxf(f1, 0.f);
          }
          return pack_bf16x2(f0, f1);
        };
        const uint32_t pk = tmem + kPackCol + (static_cast<uint32_t>(q * 32) << 16);
        if (kDrain) {
          // drain: bias, ReLU and rounding here, then the accumulator is free for the
          // next tile's MMAs while the stores below run
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32], w[16];
            tc_ld_32x32b_x32_wait(acc + c * 32, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = act_pair(v[2 * i], v[2 * i + 1]);
            tc_st_32x32b_x16(pk + c * 16, w);
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) arrive_cluster(leader_addr(&acc_empty[b]));
        }
        uint32_t* stage32 = reinterpret_cast<uint32_t*>(stage);
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t w[16];
          if (kDrain) {
            tc_ld_32x32b_x16_wait(pk + c * 16, w);
          } else {
            uint32_t v[32];
            tc_ld_32x32b_x32_wait(acc + c * 32, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = act_pair(v[2 * i], v[2 * i + 1]);
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) stage32[i * 32 + (lane ^ ((i & 7) << 2))] = w[i];
          __syncwarp();
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const int i = r * 8 + (lane >> 2);
            const int sw = (i & 7) << 2;
            const uint4 a = *reinterpret_cast<const uint4*>(stage32 + i * 32 + (((lane & 3) * 8) ^ sw));
            const uint4 e = *reinterpret_cast<const uint4*>(stage32 + i * 32 + (((lane & 3) * 8 + 4) ^ sw));
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t sel = h ? 0x7632u : 0x5410u;  // token 2i + h: high or low halves
              uint4 x = make_uint4(__byte_perm(a.x, a.y, sel), __byte_perm(a.z, a.w, sel),
                                   __byte_perm(e.x, e.y, sel), __byte_perm(e.z, e.w, sel));
              const int j = 2 * i + h;
              const int m = tb * BN + c * 32 + j;
              const int n = n_piece;
              const bool valid = m < p.rowsB && n < p.rowsA;
              if (valid && kEpi != kEpiFull) {
                *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(m) * p.ldo + n) = x;
              } else if (valid) {
                if (p.gate) {
                  const uint32_t gb = (gstage[c * 32 + j] >> (8 * (lane & 3))) & 0xFFu;
                  apply_gate(x, gb);
                }
                if (p.a24_vals) {
                  const uint32_t n0 = pick2_nibble(x.x, x.y);
                  const uint32_t n1 = pick2_nibble(x.z, x.w);
                  const uint32_t k0 = kept_pair(x.x, x.y, n0);
                  const uint32_t k1 = kept_pair(x.z, x.w, n1);
                  mask_group(x.x, x.y, n0);
                  mask_group(x.z, x.w, n1);
                  *reinterpret_cast<uint2*>(p.a24_vals + static_cast<int64_t>(m) * p.a24_ldv + n / 2) =
                      make_uint2(k0, k1);
                  p.a24_meta[static_cast<int64_t>(m) * p.a24_ldm + n / 8] = static_cast<uint8_t>(n0 | (n1 << 4));
                }
                if (p.dbias) {
                  const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                  for (int k = 0; k < 4; ++k) {
                    dsum[2 * k] += __uint_as_float(xw[k] << 16);
                    dsum[2 * k + 1] += __uint_as_float(xw[k] & 0xFFFF0000u);
                  }
                }
                *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(m) * p.ldo + n) = x;
              }
            }
          }
          __syncwarp();
        }
      } else {
        // out[a_row, j]: A row = token, B row = output feature
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tc_ld_32x32b_x32_wait(acc + c * 32, v);
          const int n0 = tb * BN + c * 32;
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float f0 = __uint_as_float(v[2 * j]), f1 = __uint_as_float(v[2 * j + 1]);
            if (p.bias) {
              f0 += (n0 + 2 * j < p.rowsB) ? p.bias[n0 + 2 * j] : 0.f;
              f1 += (n0 + 2 * j + 1 < p.rowsB) ? p.bias[n0 + 2 * j + 1] : 0.f;
            }
            if (p.relu) {
              f0 = fmaxf(f0, 0.f);
              f1 = fmaxf(f1, 0.f);
            }
            w[j] = pack_bf16x2(f0, f1);
          }
          if (a_row < p.rowsA) {
            __nv_bfloat16* o = p.out + static_cast<int64_t>(a_row) * p.ldo + n0;
#pragma unroll
            for (int pc = 0; pc < 4; ++pc)
              if (n0 + pc * 8 < p.rowsB)
                *reinterpret_cast<uint4*>(o + pc * 8) =
                    make_uint4(w[4 * pc], w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
          }
        }
      }
      if (!kDrain) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_cluster(leader_addr(&acc_empty[b]));
      }
      if (kTransOut && kEpi == kEpiFull && p.dbias) {
        // lanes l, l ^ 4, ..., l ^ 28 hold the same 8 features: sum them, then one
        // fp32 atomic per feature and tile
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          dsum[i] += __shfl_xor_sync(0xffffffffu, dsum[i], 4);
          dsum[i] += __shfl_xor_sync(0xffffffffu, dsum[i], 8);
          dsum[i] += __shfl_xor_sync(0xffffffffu, dsum[i], 16);
        }
        if (lane < 4) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            if (n_piece + i < p.rowsA) atomicAdd(p.dbias + n_piece + i, dsum[i]);
        }
      }
    }
  }

  tc_fence_before();
  cluster_sync();  // the peer may still signal this CTA's barriers until here
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// ---------------------------------------------------------------- masked dW GEMM (CTA pair)
// A cluster of 2 CTAs computes each 256 x 256 tile of dW with pair MMAs
// (tcgen05.mma.cta_group::2, M = 256, N = 256, K = 16). CTA c of the pair holds
// dW rows 128c..128c+127 of the tile (its A operand: dY's 128 features) and
// columns 128c..128c+127 of the tile's B operand (X's columns), so each SM stages
// and reads only half of B; CTA 0 (the leader) issues the MMAs and both CTAs'
// loads complete on its `full` barrier. Each CTA's TMEM receives the accumulator
// rows of its own 128 dW rows. Per stage (64 tokens) per CTA: A = dY [64 tokens x
// 128 features] and B = X [64 tokens x 128 columns], each as two 64-wide boxes
// (128 B rows, 128B swizzle), MN-major for both operands.
template <int STAGES>
struct DwSmem {
  static constexpr int kA = 64 * 128 * 2;
  static constexpr int kB = 64 * 128 * 2;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kA;
  // spare bytes after the last B stage: a B descriptor covers this CTA's 128
  // columns, and the pad keeps even a read of the full 256 inside the allocation
  static constexpr int kPad = 2 * 8192;
  // epilogue staging: per epilogue warp 32 dW rows x 64 columns of bf16 (4 KB)
  static constexpr int kOffStage = kOffB + STAGES * kB + kPad;
  static constexpr int kStage = 32 * 64 * 2;
  static constexpr int kOffBar = kOffStage + 4 * kStage;
  static constexpr int kBytes = kOffBar + 8 * (2 * STAGES + 5) + 16;
  static constexpr int kTxPair = 2 * (kA + kB);  // both CTAs' A and B, counted on the leader's barrier
};

template <int STAGES, bool kMasked>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    dw_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2, const DwParams p) {
  using L = DwSmem<STAGES>;
  constexpr int BN = 256;
  constexpr uint32_t kIdesc = idesc_bf16(2 * kBM, BN, false, /*a_mn=*/true, /*b_mn=*/true);
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // keeps shared (not generic) accesses
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBar);  // leader's is used
  uint64_t* empty = full + STAGES;                                    // leader's commit, both CTAs
  uint64_t* acc_full = empty + STAGES;                                // [2] leader's commit, both CTAs
  uint64_t* acc_empty = acc_full + 2;                                 // [2] leader's is used (8 arrivals)
  uint64_t* spare = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(spare + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 8);  // 4 epilogue warps x 2 CTAs
    }
    mbar_init(spare, 1);
    *abort_flag = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (p.tilesA_main < p.tilesA) tma_prefetch_desc(&tmA2);
    if (p.tilesB_main < p.tilesB) tma_prefetch_desc(&tmB2);
  }
  if (warp == 1) {  // pair allocation: one warp of each CTA, same columns in both
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(512)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int rank = static_cast<int>(cluster_ctarank());
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  pdl_wait();  // the previous kernel's outputs (under programmatic launch)
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl) {
        int ta, tb;
        tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
        // extra tiles read the second operands, from their first row / column
        const bool xa = ta >= p.tilesA_main, xb = tb >= p.tilesB_main;
        const CUtensorMap* ma = xa ? &tmA2 : &tmA;
        const CUtensorMap* mb = xb ? &tmB2 : &tmB;
        const int a0 = (2 * (xa ? ta - p.tilesA_main : ta) + rank) * kBM;
        const int b0 = (xb ? tb - p.tilesB_main : tb) * BN + rank * (BN / 2);
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!p24_wait(&empty[s], ph ^ 1, abort_flag, p.status)) { ok = false; break; }
          if (leader) mbar_arrive_expect_tx(&full[s], L::kTxPair);
          const uint32_t fullL = leader_addr(&full[s]);
          uint8_t* a = smem + L::kOffA + s * L::kA;
          uint8_t* b = smem + L::kOffB + s * L::kB;
          for (int i = 0; i < 2; ++i) tma_load_2d_pair(a + i * 8192, ma, fullL, a0 + i * 64, kb * 64);
          for (int i = 0; i < 2; ++i) tma_load_2d_pair(b + i * 8192, mb, fullL, b0 + i * 64, kb * 64);
        }
      }
      // Drain: the last issued loads must land before the CTA may exit.
      const uint32_t n_drain = it < STAGES ? it : STAGES;
      for (uint32_t i = 0; i < n_drain; ++i) {
        const uint32_t j = it - 1 - i;
        if (leader) p24_wait_quiet(&full[j % STAGES], (j / STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer (leader CTA only)
    if (leader) {
      uint32_t it = 0, tl = 0;
      bool ok = true;
      for (int t = cid; t < p.num_tiles && ok; t += ncl, ++tl) {
        const int b = tl & 1;
        const uint32_t aph = (tl >> 1) & 1;
        if (!p24_wait(&acc_empty[b], aph ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + b * BN;
        for (int kb = 0; kb < p.nkb; ++kb, ++it) {
          const int s = it % STAGES;
          const uint32_t ph = (it / STAGES) & 1;
          if (!p24_wait(&full[s], ph, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t a_base = smem_u32(smem + L::kOffA + s * L::kA);
            const uint32_t b_base = smem_u32(smem + L::kOffB + s * L::kB);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc(a_base + kk * 2048, 8192, 1024, kSwizzle128B);
              const uint64_t bdesc = smem_desc(b_base + kk * 2048, 8192, 1024, kSwizzle128B);
              tc_mma_pair(d_tmem, adesc, bdesc, kIdesc, (kb | kk) != 0);
            }
            tc_commit_pair(&empty[s], 0x3);
          }
          __syncwarp();
        }
        if (!ok) break;
        if (lane == 0) tc_commit_pair(&acc_full[b], 0x3);
        __syncwarp();
      }
      // Make sure no MMA is still running before TMEM is released.
      if (lane == 0) {
        tc_commit_pair(spare, 0x1);
        p24_wait_quiet(spare, 0);
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------ epilogue (warps 2-5, both CTAs)
    const int q = warp & 3;
    uint32_t tl = 0;
    for (int t = cid; t < p.num_tiles; t += ncl, ++tl) {
      int ta, tb;
      tile_coords(t, p.tilesA, p.tilesB, p.group, ta, tb);
      const bool extra = ta >= p.tilesA_main || tb >= p.tilesB_main;
      const int b = tl & 1;
      const uint32_t aph = (tl >> 1) & 1;
      // The mask bytes of this thread's dW row in the tile (8 columns a byte), read
      // while the tile's main loop still runs, so that no load sits in the epilogue.
      uint32_t mwc[BN / 32] = {};
      if constexpr (kMasked) {
        if (!extra) {
          const int n = (2 * ta + rank) * kBM + q * 32 + lane;
          const int kb0 = tb * BN / 8;  // first mask byte of the tile
          if (n < p.N) {
            const uint8_t* mrow = p.meta + static_cast<int64_t>(n) * p.ldm + kb0;
            if (kb0 + BN / 8 <= p.ldm) {
#pragma unroll
              for (int h = 0; h < BN / 128; ++h) {
                const uint4 x = *reinterpret_cast<const uint4*>(mrow + 16 * h);
                mwc[4 * h] = x.x;
                mwc[4 * h + 1] = x.y;
                mwc[4 * h + 2] = x.z;
                mwc[4 * h + 3] = x.w;
              }
            } else {
#pragma unroll
              for (int i = 0; i < BN / 8; ++i)
                if (kb0 + i < p.ldm) mwc[i / 4] |= static_cast<uint32_t>(mrow[i]) << (8 * (i % 4));
            }
          }
        }
      }
      if (!p24_wait(&acc_full[b], aph, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t acc = tmem + b * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (extra) {
        // unmasked rows / columns of the second output
        const int n2 = (2 * (ta >= p.tilesA_main ? ta - p.tilesA_main : ta) + rank) * kBM + q * 32 + lane;
        const int kbase = (tb >= p.tilesB_main ? tb - p.tilesB_main : tb) * BN;
        const int nlim = ta >= p.tilesA_main ? p.N2 : p.N;
        const int klim = tb >= p.tilesB_main ? p.K2 : p.K;
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tc_ld_32x32b_x32_wait(acc + c * 32, v);
          const int k0 = kbase + c * 32;
          if (n2 < nlim && k0 < klim) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
            __nv_bfloat16* o = p.out2 + static_cast<int64_t>(n2) * p.ldo2 + k0;
#pragma unroll
            for (int pc = 0; pc < 4; ++pc)
              if (k0 + pc * 8 < klim)
                *reinterpret_cast<uint4*>(o + pc * 8) = make_uint4(w[4 * pc], w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_cluster(leader_addr(&acc_empty[b]));
        continue;
      }
      ta = 2 * ta + rank;
      // Thread = dW row ta * kBM + q * 32 + lane (its TMEM lane). Two 32-column chunks of
      // the warp's 32 rows go through a 32 x 64 shared-memory stage (16-byte pieces
      // XOR-swizzled by row: the row writes and the line reads are both free of bank
      // conflicts), so that each store instruction writes 4 rows x 128 bytes.
      const int row0 = ta * kBM + q * 32;
      uint8_t* stg = smem + L::kOffStage + q * L::kStage;
      for (int cp = 0; cp < BN / 64; ++cp) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * cp + h;
          uint32_t v[32];
          tc_ld_32x32b_x32_wait(acc + c * 32, v);
          uint32_t w[16];
          if constexpr (kMasked) {
            // bytes past the last column are padding (0x44) or unread: their groups are
            // past K, so no store reads them
            uint32_t mw = mwc[0];  // mwc[c] by selects: the words stay in registers
#pragma unroll
            for (int i = 1; i < BN / 32; ++i) mw = (c == i) ? mwc[i] : mw;
#pragma unroll
            for (int g = 0; g < 8; ++g) {
              const uint32_t nib = (mw >> (4 * g)) & 0xFu;
              const uint32_t kbits = (1u << (nib & 3u)) | (1u << (nib >> 2));
              float f[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) f[i] = (kbits >> i) & 1u ? __uint_as_float(v[4 * g + i]) : 0.f;
              w[2 * g] = pack_bf16x2(f[0], f[1]);
              w[2 * g + 1] = pack_bf16x2(f[2], f[3]);
            }
          } else {
#pragma unroll
            for (int k = 0; k < 16; ++k) w[k] = pack_bf16x2(__uint_as_float(v[2 * k]), __uint_as_float(v[2 * k + 1]));
          }
#pragma unroll
          for (int pc = 0; pc < 4; ++pc)
            *reinterpret_cast<uint4*>(stg + lane * 128 + (((4 * h + pc) ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * pc], w[4 * pc + 1], w[4 * pc + 2], w[4 * pc + 3]);
        }
        __syncwarp();
        const int kc = tb * BN + cp * 64 + (lane & 7) * 8;  // this lane's 8 columns
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int row = 4 * r + (lane >> 3);
          const uint4 x = *reinterpret_cast<const uint4*>(stg + row * 128 + (((lane & 7) ^ (row & 7)) << 4));
          if (row0 + row < p.N && kc < p.K)
            *reinterpret_cast<uint4*>(p.out + static_cast<int64_t>(row0 + row) * p.ldo + kc) = x;
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_cluster(leader_addr(&acc_empty[b]));
    }
  }

  tc_fence_before();
  cluster_sync();  // the peer may still signal this CTA's barriers until here
  tc_fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512) : "memory");
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D view {64, rows, K/64} of a row-major [rows, K] bf16 matrix (K % 64 == 0), so
// that one box {64, box_rows, 2} is a 128-K slab laid out as two 64-K halves.
bool make_map_kslab(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t row_bytes,
                    uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, rows, K / 64};
  cuuint64_t strides[2] = {row_bytes, 128};
  cuuint32_t box[3] = {64, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
                 uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  (void)elem_bytes;
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Clusters of `cluster` CTAs of this kernel that can be resident at once (GPCs
// need not divide evenly into clusters, so this can be below SMs / cluster).
// A persistent grid larger than this would leave whole clusters for a second wave.
constexpr int kMaxDevices = 64;

template <class Kern>
int max_active_clusters(Kern kern, int cluster, int threads, int smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cluster), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = static_cast<unsigned>(cluster);
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
    cudaGetLastError();  // clear; fall back to the SM count
    return 0;
  }
  return n;
}

// Per-device launch setup of one kernel instantiation: its dynamic shared memory
// attribute set once, and the number of co-resident clusters (0: query failed, use
// SMs / 2). Kept per device, computed on the first launch there.
struct LaunchSetup {
  std::once_flag once[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
  int clusters[kMaxDevices] = {};
};

template <class Kern>
cudaError_t launch_setup(LaunchSetup& ls, Kern kern, int cluster, int threads, int smem, int& clusters) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::call_once(ls.once[dev], [&] {
    ls.err[dev] = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (ls.err[dev] == cudaSuccess) ls.clusters[dev] = max_active_clusters(kern, cluster, threads, smem);
  });
  clusters = ls.clusters[dev];
  return ls.err[dev];
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

// Sparse tile widths: N = 256 (one TMEM accumulator, the most MMA work buffered
// per shared-memory byte, the epilogue overlapped through the drained copy below),
// except for plain epilogues with very short main loops, which take N = 192 with two
// accumulators. The ReLU' gate turns into bits while the tile's main loop runs,
// before the accumulator is ready.
constexpr int kSpBNWide = 256;
constexpr int kSpBNOverlap = 192;
// The drained epilogue (one accumulator): the tile is copied out of the accumulator
// as bf16 pairs and released before its stores, which then overlap the next tile's main
// loop (70B step: up forward -5%, gated dH -8%; 7B gated dH -14%). A gated tile's gate
// words are read after those stores, so at short K the next main loop ends first and
// the drain loses (1.3B dH, K = 2048: +9%); gated tiles drain from this many K-blocks.
#ifndef P24_DRAIN_GATE_MIN_NKB
#define P24_DRAIN_GATE_MIN_NKB 32
#endif
#ifndef P24_OVERLAP_MAX_NKB
#define P24_OVERLAP_MAX_NKB 8  // K-blocks (of 128) up to which plain epilogues take the two-accumulator tile
#endif
constexpr int kSpStages = 4;
constexpr int kDwStages = 6;

template <int BN, bool kTrans, int kEpi, bool kGather = false, bool kDrainOk = true>
cudaError_t run_spmm(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& e, const CUtensorMap& l,
                     const CUtensorMap& t, const SpmmParams& p, cudaStream_t s) {
  using L = SpmmSmem<BN, kSpStages>;
  auto kern = spmm_kernel<BN, kSpStages, kTrans, kEpi, kGather, kDrainOk>;
  const int smem = L::kBytes + 1024;
  constexpr int kThreads = kGather ? 320 + kGatherThreads : 320;  // + the gather warps
  static LaunchSetup setup;
  int clusters = 0;
  cudaError_t err = launch_setup(setup, kern, 2, kThreads, smem, clusters);
  if (err != cudaSuccess) return err;
  if (clusters == 0) clusters = num_sms() / 2;
  const int grid = 2 * std::min(p.num_tiles, clusters);  // clusters of 2, all resident
  err = launch_pdl(kern, dim3(grid), dim3(kThreads), smem, s, a, b, e, l, t, p);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaGetLastError();
}

}  // namespace

bool make_tensor_map_2d(CUtensorMap* m, bool bf16, const void* base, uint64_t inner, uint64_t outer,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, bool swizzle128) {
  return make_map_2d(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, bf16 ? 2 : 1, base,
                     inner, outer, row_bytes, box_inner, box_outer,
                     swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

cudaError_t launch_spmm(const p24_sparse& A, const void* B, int64_t rowsB, int64_t ldb, void* out, int64_t ldo,
                        bool transposed_out, const EpiArgs& epi, int* status, cudaStream_t s) {
  if (A.rows == 0 || rowsB == 0) return cudaSuccess;
  const bool heavy_epilogue = epi.act24.vals != nullptr;
  // Two accumulators at the narrower tile only for plain epilogues of very short main
  // loops (GPT-2, K = 768). Measured against N = 256 with the drained epilogue: the 1.3B
  // up forward (K = 2048) is 12% faster on N = 256, the 7B up forward with the 2:4
  // activation prune 17% faster, GPT-2 1% slower.
  const bool overlap = transposed_out && !heavy_epilogue && !epi.gate && !epi.dbias &&
                       (A.cols + 127) / 128 <= P24_OVERLAP_MAX_NKB;
  const int BN = overlap ? kSpBNOverlap : kSpBNWide;
  SpmmParams p{};
  p.rowsA = static_cast<int>(A.rows);
  p.rowsB = static_cast<int>(rowsB);
  p.K = static_cast<int>(A.cols);
  p.tilesA = static_cast<int>((A.rows + 2 * kBM - 1) / (2 * kBM));  // A tile pairs (one per cluster)
  p.tilesB = static_cast<int>((rowsB + BN - 1) / BN);
  p.num_tiles = p.tilesA * p.tilesB;
  // 16 A-tile pairs per raster group: with 76 pairs resident, a wave covers about
  // 16 A x 5 B tiles, close to the shape that needs the fewest panel bytes per wave
  // (a B panel, 256 x K bf16, is 1.78x a compressed A panel). Measured on the 70B
  // step: 8 and 12 along A, and 8 along B, within 1%; 16 or 32 along B, 2-5% slower.
  p.group = std::min(p.tilesA, 16);
  p.nkb = static_cast<int>((A.cols + 127) / 128);
  p.out = static_cast<__nv_bfloat16*>(out);
  p.ldo = ldo;
  p.bias = epi.bias;
  p.relu = epi.relu ? 1 : 0;
  p.gate = static_cast<const uint16_t*>(epi.gate);
  p.ldg = epi.ldg;
  p.dbias = epi.dbias;
  p.stall_stage = epi.test_stall ? 3 : 0;
  if (!transposed_out && (epi.gate || epi.dbias)) return cudaErrorInvalidValue;
  p.a24_vals = static_cast<uint16_t*>(epi.act24.vals);
  p.a24_ldv = epi.act24.ldv;
  p.a24_meta = epi.act24.meta;
  p.a24_ldm = epi.act24.ldm;
  p.status = status;
  if (A.cols == 0) return cudaErrorInvalidValue;

  CUtensorMap ta, tb, te;
  // K % 64 == 0: one 3-D load per stage for B; otherwise two 2-D loads, whose out-of-range
  // part past K is zero-filled (a 3-D view would read the next row there).
  p.b3d = (A.cols % 64 == 0) ? 1 : 0;
  const bool b_ok = p.b3d ? make_map_kslab(&tb, B, A.cols, rowsB, ldb * 2, BN / 2)
                          : make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, A.cols, rowsB, ldb * 2, 64,
                                        BN / 2, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A.vals, A.cols / 2, A.rows, A.ldv * 2, 64, kBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !b_ok ||
      !make_map_2d(&te, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A.meta, A.ldm, A.rows, A.ldm, 16 * kEStages, kBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  // low-rank term: dense stages after the sparse ones (a copy of A's map when there is none)
  CUtensorMap tl = ta, tt = ta;
  if (epi.lr_r > 0) {
    if (!epi.lr_a || !epi.lr_b) return cudaErrorInvalidValue;
    p.nad = static_cast<int>((epi.lr_r + 63) / 64);
    if (!make_map_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, epi.lr_a, epi.lr_r, A.rows, epi.lr_lda * 2, 64, kBM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map_2d(&tt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, epi.lr_b, epi.lr_r, rowsB, epi.lr_ldb * 2, 64, BN / 2,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return cudaErrorInvalidValue;
  }
  if (!transposed_out) {
    if (heavy_epilogue) return cudaErrorInvalidValue;  // the activation prune is transposed-only
    return run_spmm<kSpBNWide, false, kEpiStore>(ta, tb, te, tl, tt, p, s);
  }
  if (heavy_epilogue || epi.gate || epi.dbias) {
    return (!epi.gate || p.nkb >= P24_DRAIN_GATE_MIN_NKB)
               ? run_spmm<kSpBNWide, true, kEpiFull>(ta, tb, te, tl, tt, p, s)
               : run_spmm<kSpBNWide, true, kEpiFull, false, false>(ta, tb, te, tl, tt, p, s);
  }
  return overlap ? run_spmm<kSpBNOverlap, true, kEpiStore>(ta, tb, te, tl, tt, p, s)
                 : run_spmm<kSpBNWide, true, kEpiStore>(ta, tb, te, tl, tt, p, s);
}

cudaError_t launch_gemm_nt(const void* A, int64_t M, int64_t lda, const void* B, int64_t N, int64_t ldb, int64_t K,
                           void* C, int64_t ldc, int* status, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (K == 0) return cudaMemset2DAsync(C, ldc * 2, 0, N * 2, M, s);
  // the sparse GEMM's pipeline with only dense stages: A as the low-rank A_l, B as B_l
  SpmmParams p{};
  p.rowsA = static_cast<int>(M);
  p.rowsB = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.tilesA = static_cast<int>((M + 2 * kBM - 1) / (2 * kBM));
  p.tilesB = static_cast<int>((N + kSpBNWide - 1) / kSpBNWide);
  p.num_tiles = p.tilesA * p.tilesB;
  p.group = std::min(p.tilesA, 16);
  p.nkb = 0;
  p.nad = static_cast<int>((K + 63) / 64);
  p.out = static_cast<__nv_bfloat16*>(C);
  p.ldo = ldc;
  p.status = status;
  CUtensorMap tl, tt;
  if (!make_map_2d(&tl, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, lda * 2, 64, kBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&tt, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, ldb * 2, 64, kSpBNWide / 2,
                   CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  return run_spmm<kSpBNWide, false, kEpiStore>(tl, tt, tl, tl, tt, p, s);
}

cudaError_t launch_vnm_spmm(const uint8_t* colidx, const p24_sparse& A, int V, int Mg, const void* B, int64_t N,
                            int64_t ldb, const float* bias, bool relu, void* Y, int64_t ldy, int* status,
                            cudaStream_t s) {
  if (A.rows == 0 || N == 0) return cudaSuccess;
  // the caller checked: V % 256 == 0, condensed K % 128 == 0, N % 256 == 0
  const int64_t K = A.cols / 4 * Mg;  // logical reduction length (rows of B)
  SpmmParams p{};
  p.rowsA = static_cast<int>(A.rows);
  p.rowsB = static_cast<int>(N);
  p.K = static_cast<int>(A.cols);
  p.tilesA = static_cast<int>((A.rows + 2 * kBM - 1) / (2 * kBM));
  p.tilesB = static_cast<int>(N / kSpBNWide);
  p.num_tiles = p.tilesA * p.tilesB;
  p.group = std::min(p.tilesA, 16);
  p.nkb = static_cast<int>(A.cols / 128);
  p.out = static_cast<__nv_bfloat16*>(Y);
  p.ldo = ldy;
  p.bias = bias;
  p.relu = relu ? 1 : 0;
  p.status = status;
  p.vnm_cix = reinterpret_cast<const uint32_t*>(colidx);
  p.vnm_group = Mg;
  p.vnm_V = V;
  p.vnm_G = static_cast<int>(K / Mg);
  p.vnm_K = static_cast<int>(K);
  p.vnm_B = static_cast<const uint16_t*>(B);
  p.vnm_ldb = ldb;
  CUtensorMap ta, tb, te;
  if (!make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A.vals, A.cols / 2, A.rows, A.ldv * 2, 64, kBM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&te, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A.meta, A.ldm, A.rows, A.ldm, 16 * kEStages, kBM,
                   CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  tb = ta;  // B is gathered by the kernel's threads (p.vnm_B), not by TMA
  return run_spmm<kSpBNWide, false, kEpiStore, true>(ta, tb, te, ta, tb, p, s);
}

namespace {
cudaError_t run_dw(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N, int64_t K,
                   const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw, const DwExtra& ex, int* status,
                   cudaStream_t s);
}

cudaError_t launch_masked_dw(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N,
                             int64_t K, const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw, int* status,
                             cudaStream_t s) {
  if (!meta) return cudaErrorInvalidValue;
  return run_dw(dY, lddy, X, ldx, M, N, K, meta, ldm, dW, lddw, DwExtra{}, status, s);
}

cudaError_t launch_masked_dw_extra(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N,
                                   int64_t K, const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw,
                                   const DwExtra& ex, int* status, cudaStream_t s) {
  if (!meta || !ex.out2 || (ex.a2 != nullptr) == (ex.b2 != nullptr)) return cudaErrorInvalidValue;
  return run_dw(dY, lddy, X, ldx, M, N, K, meta, ldm, dW, lddw, ex, status, s);
}

cudaError_t launch_gemm_tn(const void* A, int64_t lda, const void* B, int64_t ldb, int64_t M, int64_t N, int64_t K,
                           void* C, int64_t ldc, int* status, cudaStream_t s) {
  return run_dw(A, lda, B, ldb, M, N, K, nullptr, 0, C, ldc, DwExtra{}, status, s);
}

namespace {
cudaError_t run_dw(const void* dY, int64_t lddy, const void* X, int64_t ldx, int64_t M, int64_t N, int64_t K,
                   const uint8_t* meta, int64_t ldm, void* dW, int64_t lddw, const DwExtra& ex, int* status,
                   cudaStream_t s) {
  if (N == 0 || K == 0) return cudaSuccess;
  if (M == 0) {
    // empty reduction: dW = 0 everywhere
    if (ex.a2 && ex.n2 > 0) {
      cudaError_t e = cudaMemset2DAsync(ex.out2, ex.ldo2 * 2, 0, K * 2, ex.n2, s);
      if (e != cudaSuccess) return e;
    }
    if (ex.b2 && ex.k2 > 0) {
      cudaError_t e = cudaMemset2DAsync(ex.out2, ex.ldo2 * 2, 0, ex.k2 * 2, N, s);
      if (e != cudaSuccess) return e;
    }
    return cudaMemset2DAsync(dW, lddw * 2, 0, K * 2, N, s);
  }
  DwParams p{};
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.M = static_cast<int>(M);
  p.tilesA_main = static_cast<int>((N + 2 * kBM - 1) / (2 * kBM));  // A tile pairs (one per cluster)
  p.tilesB_main = static_cast<int>((K + 255) / 256);
  p.tilesA = p.tilesA_main + (ex.a2 ? static_cast<int>((ex.n2 + 2 * kBM - 1) / (2 * kBM)) : 0);
  p.tilesB = p.tilesB_main + (ex.b2 ? static_cast<int>((ex.k2 + 255) / 256) : 0);
  p.num_tiles = p.tilesA * p.tilesB;
  // groups of at most 8 A-tile pairs, evened out so that extra A tiles join main ones
  p.group = (p.tilesA + (p.tilesA + 7) / 8 - 1) / ((p.tilesA + 7) / 8);
  p.nkb = static_cast<int>((M + 63) / 64);
  p.out = static_cast<__nv_bfloat16*>(dW);
  p.ldo = lddw;
  p.meta = meta;
  p.ldm = ldm;
  p.status = status;
  p.N2 = static_cast<int>(ex.n2);
  p.K2 = static_cast<int>(ex.k2);
  p.out2 = static_cast<__nv_bfloat16*>(ex.out2);
  p.ldo2 = ex.ldo2;
  CUtensorMap ta, tb, ta2, tb2;
  if (!make_map_2d(&ta, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dY, N, M, lddy * 2, 64, 64,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map_2d(&tb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, X, K, M, ldx * 2, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  ta2 = ta;
  tb2 = tb;
  if ((ex.a2 && !make_map_2d(&ta2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ex.a2, ex.n2, M, ex.lda2 * 2, 64, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B)) ||
      (ex.b2 && !make_map_2d(&tb2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ex.b2, ex.k2, M, ex.ldb2 * 2, 64, 64,
                             CU_TENSOR_MAP_SWIZZLE_128B)))
    return cudaErrorInvalidValue;
  using L = DwSmem<kDwStages>;
  auto kern = meta ? dw_kernel<kDwStages, true> : dw_kernel<kDwStages, false>;
  const int smem = L::kBytes + 1024;
  static LaunchSetup setup_masked, setup_plain;
  int clusters = 0;
  cudaError_t err = launch_setup(meta ? setup_masked : setup_plain, kern, 2, 192, smem, clusters);
  if (err != cudaSuccess) return err;
  if (clusters == 0) clusters = num_sms() / 2;
  const int grid = 2 * std::min(p.num_tiles, clusters);  // clusters of 2, all resident
  err = launch_pdl(kern, dim3(grid), dim3(192), smem, s, ta, tb, ta2, tb2, p);
  if (err != cudaSuccess) return err;
  count_launch();
  return cudaGetLastError();
}
}  // namespace

}  // namespace p24
