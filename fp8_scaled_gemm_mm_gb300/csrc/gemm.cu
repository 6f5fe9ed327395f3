// gemm.cu -- E4M3 x E4M3 scaled GEMM on sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Computes out[m,n] = round(a_s * b_s * sum_k A[m,k] B[n,k] (+ bias[n])), the rowwise /
// per-tensor scaled FP8 GEMM of sglang PR #34318 ("[Kernel] Route large SM90
// row/column-scaled FP8 GEMMs to Torch", Summary) and of the prhub summary of
// sglang PR #33148 (per-tensor scalar scales used as they are, weight [N,K] K-major).
//
// One persistent CTA per SM (192 threads), warp-specialized:
//   warp 0      TMA producer: A [128 x 128] and B [BN x 128] byte tiles, 128-byte
//               swizzle, into a STAGES-deep shared-memory ring (full/empty mbarriers).
//               Out-of-bounds rows and the K tail arrive as zeros.
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=BN, K=32 per
//               instruction, fp32 accumulate) from one thread; tcgen05.commit frees
//               each stage and publishes each finished accumulator.
//   warps 2..5  epilogue: tcgen05.ld 32 columns at a time, scale (and bias), round to
//               bf16/fp16, stage in swizzled shared memory, TMA store (edges clipped).
// Two TMEM accumulators alternate so that the epilogue of tile i overlaps the
// mainloop of tile i+1.  Tiles are visited in groups of `raster` M-blocks (sized
// from K so that a group's A panel stays in L2) so that the CTAs running at the
// same time share A and B panels in L2.
//
// The tile width (BN = 256, 128 or 64) is the one with the smallest estimated time,
// waves x width / the width's relative MMA efficiency.
//
// Per-group A scales (one per 128-wide K block, the layout the group quant produces),
// optionally with 128 x 128 block B scales, run in fp8_gemm_group_kernel: every K
// block goes to its own TMEM accumulator (128 x 256 tiles, a ring of two) and eight
// epilogue warps, given the registers of the TMA/MMA warpgroup by setmaxnreg, fold it
// in: acc += a_s[m, kb] (* b_s[n/128, kb]) * partial_kb, in fp32 registers.
//
// M <= 128 (outside deterministic mode) runs fp8_gemm_swap_splitk_kernel: the weight
// is the MMA's 128-row operand and K is split over a thread-block cluster whose
// partials are summed in rank order through distributed shared memory.
//
// Deterministic mode picks the tile from N alone, uses one instruction shape and the
// natural K-block order for every problem, with no split of K, so row m of the result
// does not depend on M or on the other rows (sglang PR #44861, Modifications: fixed
// N=64/K=128 reduction tiles, zero-filled K tails).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace fp8mm {
namespace {

constexpr int BM = 128;
constexpr int BK = 128;           // K elements (= bytes) per stage: one 128-byte swizzle row
constexpr int UMMA_K = 32;        // K per tcgen05.mma for 8-bit operands
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;

struct GemmArgs {
  int M, N, K;
  int num_kb;
  int m_blocks, n_blocks, tiles;
  int raster;
  int a_mode, b_mode;
  int64_t a_ld;
  int64_t b_ld;   // block B scales: blocks per row of blocks (K / 128)
  const float* a_scale;
  const float* b_scale;
  const __nv_bfloat16* bias;
  int out_fp16;
  int det_splits;   // deterministic mode: K ranges summed in order (1 = no split)
  int* status;
  // Limit of the pipeline's waits (stage, accumulator and cluster hand-offs).  The
  // drains -- a producer waiting for its last loads, the MMA thread for its last
  // MMAs -- always keep the full kWaitTimeoutNs: every copy and MMA in flight must
  // have landed before a CTA releases TMEM or exits, whatever this limit is.
  uint64_t timeout_ns;
};

// First K block of range r of the deterministic split (range r is [kb_begin(r), kb_begin(r + 1))).
__host__ __device__ __forceinline__ int det_kb_begin(int r, int num_kb, int splits) {
  return static_cast<int>(static_cast<int64_t>(r) * num_kb / splits);
}

// The deterministic mode's output value: ((acc * a_s) * b_s) + bias, each step rounded
// once (no contraction), so that the cluster kernel and the fold kernel of that mode
// produce the same bits from the same fp32 sum.
__device__ __forceinline__ float det_out(float acc, float sa, float sb, float bias) {
  return __fadd_rn(__fmul_rn(__fmul_rn(acc, sa), sb), bias);
}

__host__ __device__ constexpr uint32_t pow2_at_least(uint32_t v) {
  uint32_t r = 32;
  while (r < v) r <<= 1;
  return r;
}

template <int BN, int STAGES>
struct Layout {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int D_BYTES = 32 * 64;  // one epilogue warp's staging buffer: 32 rows x 64 bytes
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_D = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_D + kEpiWarps * 2 * D_BYTES;
  static constexpr int NBARS = 2 * STAGES + 5;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;  // slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = pow2_at_least(2 * BN);
  static constexpr uint32_t ACC_STRIDE = TMEM_COLS / 2;   // accumulator 1 starts at a power-of-two column
  static_assert(B_BYTES % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

__device__ __forceinline__ void tile_coords(const GemmArgs& p, int t, int& mb, int& nb) {
  const int per_group = p.raster * p.n_blocks;
  const int g = t / per_group;
  const int first = g * p.raster;
  const int gsz = min(p.m_blocks - first, p.raster);
  const int r = t - g * per_group;
  mb = first + r % gsz;
  nb = r / gsz;
}

// Row scale of the rowwise / per-tensor A modes (the per-group modes run in
// fp8_gemm_group_kernel); rows past M read as 0.
__device__ __forceinline__ float a_scale_at(const GemmArgs& p, int row) {
  if (row >= p.M) return 0.0f;
  return p.a_mode == FP8MM_SCALE_A_TENSOR ? __ldg(p.a_scale) : __ldg(p.a_scale + row);
}

// fp32 value of a UE8M0 scale byte e: 2^(e-127), rounded to fp32 -- e = 0 is the
// subnormal 2^-127 (bit 22 set), e = 255 overflows to +inf (the exponent field alone).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t e) { return __uint_as_float(e ? e << 23 : 0x00400000u); }

// b_scale and bias for the 32 columns n0..n0+31 (zeros beyond N).
__device__ __forceinline__ void load_col_vectors(const GemmArgs& p, int n0, float (&sb)[32], float (&bs)[32]) {
  if (p.b_mode == 2) {   // block scales were applied per K block
#pragma unroll
    for (int j = 0; j < 32; ++j) sb[j] = 1.0f;
  } else if (p.b_mode == 0) {
    const float s = __ldg(p.b_scale);
#pragma unroll
    for (int j = 0; j < 32; ++j) sb[j] = s;
  } else if ((reinterpret_cast<uintptr_t>(p.b_scale) & 15u) == 0) {
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
      if (n0 + 4 * v < p.N) f = __ldg(reinterpret_cast<const float4*>(p.b_scale + n0) + v);
      sb[4 * v] = f.x;
      sb[4 * v + 1] = f.y;
      sb[4 * v + 2] = f.z;
      sb[4 * v + 3] = f.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) sb[j] = (n0 + j < p.N) ? __ldg(p.b_scale + n0 + j) : 0.0f;
  }
  if (p.bias == nullptr) {
#pragma unroll
    for (int j = 0; j < 32; ++j) bs[j] = 0.0f;
  } else if ((reinterpret_cast<uintptr_t>(p.bias) & 15u) == 0) {
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      uint4 u = make_uint4(0, 0, 0, 0);
      if (n0 + 8 * v < p.N) u = __ldg(reinterpret_cast<const uint4*>(p.bias + n0) + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        bs[8 * v + 2 * i] = __uint_as_float(w[i] << 16);
        bs[8 * v + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) bs[j] = (n0 + j < p.N) ? __bfloat162float(p.bias[n0 + j]) : 0.0f;
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int fp16) {
  if (fp16) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
  }
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Write one warp's 32 x 32 output block (this lane = one row) into its staging buffer
// (64-byte swizzle) and TMA-store it at column n0, row r0.  Blocks that lie wholly
// outside the output are skipped; partial ones are clipped by the TMA unit.
// Returns whether a store was issued (the caller then switches staging buffers).
__device__ __forceinline__ bool store_block(const CUtensorMap* tmD, uint8_t* buf, const uint32_t (&w)[16],
                                            int lane, int n0, int r0, int M, int N) {
  if (r0 >= M || n0 >= N) return false;
  if (lane == 0) bulk_wait_read<1>();  // the store issued from this buffer two blocks ago has read it
  __syncwarp();
  uint8_t* row = buf + lane * 64;
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(row + ((j ^ sw) << 4)) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmD, buf, n0, r0);
    bulk_commit();
  }
  return true;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmD, const GemmArgs p) {
  using L = Layout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  // 128-byte swizzle atoms and the UMMA descriptors need 1024-byte aligned shared addresses
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // A and its scales may come from the kernel launched just before this one
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int t = blockIdx.x; t < p.tiles && !*abort_flag; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
          mbar_arrive_expect_tx(&full[stage], L::A_BYTES + L::B_BYTES);
          tma_load_2d(&tmA, &full[stage], smem + L::OFF_A + stage * L::A_BYTES, kb * BK, mb * BM);
          tma_load_2d(&tmB, &full[stage], smem + L::OFF_B + stage * L::B_BYTES, kb * BK, nb * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // Every load this CTA issued must have landed before the CTA may exit.
      const int outstanding = static_cast<int>(issued < STAGES ? issued : STAGES);
      for (int j = 1; j <= outstanding; ++j) {
        int s = static_cast<int>(stage) - j;
        uint32_t ph = phase;
        if (s < 0) {
          s += STAGES;
          ph ^= 1u;
        }
        volatile int never = 0;
        mbar_wait(&full[s], ph, &never, p.status, kWaitTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      uint32_t stage = 0, phase = 0, acc_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        for (int kb = 0; ok && kb < p.num_kb; ++kb) {
          const uint32_t acc = acc_i & 1u;
          if (kb == 0) {
            ok = mbar_wait(&tempty[acc], ((acc_i >> 1) & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns);
            if (!ok) break;
            tc_fence_after();
          }
          ok = mbar_wait(&full[stage], phase, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem_base + acc * L::ACC_STRIDE;
          const uint64_t adesc = smem_desc_sw128(smem_u32(smem + L::OFF_A + stage * L::A_BYTES));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + L::OFF_B + stage * L::B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            const uint32_t accumulate = (kb | k) != 0 ? 1u : 0u;
            mma_f8f6f4(d, adesc + static_cast<uint64_t>(k * UMMA_K / 16),
                       bdesc + static_cast<uint64_t>(k * UMMA_K / 16), idesc, accumulate);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kb == p.num_kb - 1) {
            mma_commit(&tfull[acc]);
            ++acc_i;
          }
        }
      }
      // All MMAs issued here must be complete before TMEM is released.
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, p.status, kWaitTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------- epilogue
    const int ew = warp - 2;                  // staging buffer owner
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    uint8_t* stage_buf = smem + L::OFF_D + ew * 2 * L::D_BYTES;
    int dbuf = 0;
    uint32_t acc_i = 0;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int r0 = mb * BM + q * 32;
      const int nbase = nb * BN;
      const uint32_t acc = acc_i & 1u;
      if (!mbar_wait(&tfull[acc], (acc_i >> 1) & 1u, abort_flag, p.status, p.timeout_ns)) break;
      tc_fence_after();
      const float sa = a_scale_at(p, row);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(lane_addr + acc * L::ACC_STRIDE + c * 32, r);
        tmem_ld_wait();
        if (c == BN / 32 - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&tempty[acc]);
        }
        float sb[32], bs[32];
        load_col_vectors(p, nbase + c * 32, sb, bs);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float v0 = __uint_as_float(r[2 * j]) * sa * sb[2 * j] + bs[2 * j];
          const float v1 = __uint_as_float(r[2 * j + 1]) * sa * sb[2 * j + 1] + bs[2 * j + 1];
          w[j] = pack2(v0, v1, p.out_fp16);
        }
        if (store_block(&tmD, stage_buf + dbuf * L::D_BYTES, w, lane, nbase + c * 32, r0, p.M, p.N)) dbuf ^= 1;
      }
      ++acc_i;
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------- per-group A (and block B) scales
//
// The MMA cannot apply a scale that changes along K, so every 128-wide K block
// accumulates into its own TMEM buffer (a ring of NACC) and the epilogue folds it in:
// acc[m, n] += a_s[m, kb] * b_s[n / 128, kb] * partial_kb[m, n] (b_s = 1 without
// block scales).  4 x SPLIT epilogue warps share the work: warp w reads TMEM lane
// quarter w % 4 (the only one it may access) and one of SPLIT column slices of the
// tile, holding its slice of acc in fp32 registers.  The buffer is handed back to the
// MMA warp as soon as its values are in registers.
//
// Tile width matters more than anything else here: with M = 128, MMAs of N = 128
// reach about 60 % of the tensor rate on this part and N = 256 about 95 %.  So the
// preferred form is 128 x 256 with two accumulators (all 512 TMEM columns) and
// SPLIT = 2, which needs 128 accumulator registers per epilogue thread: warpgroup 0
// (TMA and MMA threads) gives its registers to the two epilogue warpgroups with
// setmaxnreg (40 / 232 of the 168 per thread the block is launched with; an SM
// sub-partition holds 16K registers and here three warps).  Without that split the
// form is 128 x 192, SPLIT = 3, 128 registers a thread.  Plain fp32 FMAs: the packed
// f32x2 form needs register pairs the TMEM loads do not produce, and the moves cost
// more than the packing saves.

// AMODE of fp8_gemm_group_kernel for the deterministic split: every K range of the
// split goes to its own accumulator and is folded by plain fp32 adds in range order;
// the A scale (per tensor or per row) comes after the sum, as in the epilogue.
constexpr int kAModeDetFold = 15;

// Columns of TMEM one tcgen05.ld brings to a per-K-block fold of the group kernel
// (64 measured 0.3-1 % faster than 32 on the block-scaled shapes: the fold is not
// bound by the load shape).
constexpr int kFoldCols = 64;

template <int BN, int STAGES, int NACC, int SPLIT, bool RS>
struct GroupLayout {
  static constexpr int EPI_WARPS = 4 * SPLIT;
  static constexpr int FIRST_EPI = RS ? 4 : 2;   // with a register split, warpgroup 0 is TMA + MMA
  static constexpr int THREADS = 32 * FIRST_EPI + 32 * EPI_WARPS;
  static constexpr int REG_LO = 40, REG_HI = 232;   // setmaxnreg values of warpgroup 0 / the others
  static constexpr int WCOLS = BN / SPLIT;   // columns of one epilogue warp
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int D_BYTES = 32 * 64;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = OFF_A + STAGES * A_BYTES;
  static constexpr int OFF_D = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = OFF_D + EPI_WARPS * 2 * D_BYTES;
  static constexpr int NBARS = 2 * STAGES + 2 * NACC + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(NACC * BN);
  static_assert(WCOLS % 32 == 0 && WCOLS <= 128 && 128 % WCOLS == 0,
                "each epilogue warp's columns must lie in one 128-column block");
  static_assert((BN * BK) % 1024 == 0, "B stage must keep 1024-byte alignment");
  static_assert(NACC * BN <= 512, "TMEM columns");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

// Scale stream of one epilogue thread for the K blocks of a tile: A scale words of
// its row (AMODE fixes the layout at compile time) and, with BBLOCK, the block B
// scale of the tile's 128 columns.  Rows past M read row M-1 and K blocks past the
// end read the last one; neither value is used.  The epilogue fetches the words of a
// group of four K blocks one group ahead and decodes them when used, so no
// arithmetic waits on a load.
template <int AMODE, bool BBLOCK>
struct ScaleStream {
  const uint32_t* a;
  int64_t a_step;   // words between consecutive K blocks (UE8M0: between groups of four)
  const float* b;
  int last;         // num_kb - 1
  __device__ __forceinline__ ScaleStream(const GemmArgs& p, int row, int nbase) {
    const int r = row < p.M ? row : p.M - 1;
    const uint32_t* base = reinterpret_cast<const uint32_t*>(p.a_scale);
    if (AMODE == FP8MM_SCALE_A_GROUP128) {
      a = base + static_cast<int64_t>(r) * p.a_ld;
      a_step = 1;
    } else {
      a = base + r;
      a_step = p.a_ld;
    }
    b = p.b_scale + static_cast<int64_t>(nbase >> 7) * p.b_ld;
    last = p.num_kb - 1;
  }
  __device__ __forceinline__ uint32_t a_raw(int kb) const {
    kb = kb < last ? kb : last;
    return __ldg(a + (AMODE == FP8MM_SCALE_A_GROUP128_UE8M0 ? (kb >> 2) : kb) * a_step);
  }
  __device__ __forceinline__ float b_raw(int kb) const {
    if (!BBLOCK) return 1.0f;
    kb = kb < last ? kb : last;
    return __ldg(b + kb);
  }
  __device__ __forceinline__ static float decode(uint32_t raw, int kb) {
    if (AMODE == FP8MM_SCALE_A_GROUP128_UE8M0) return ue8m0_to_f32((raw >> (8 * (kb & 3))) & 0xFFu);
    return __uint_as_float(raw);
  }
};

// Per-warpgroup register budgets (setmaxnreg; all four warps of the warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

template <int BN, int STAGES, int NACC, int SPLIT, bool RS, int AMODE, bool BBLOCK>
__global__ void __launch_bounds__(GroupLayout<BN, STAGES, NACC, SPLIT, RS>::THREADS, 1)
    fp8_gemm_group_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmD, const GemmArgs p) {
  using L = GroupLayout<BN, STAGES, NACC, SPLIT, RS>;
  constexpr int HALF = L::WCOLS;
  constexpr bool DET = AMODE == kAModeDetFold;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + NACC;
  uint64_t* drain = tempty + NACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], L::EPI_WARPS);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // A and its scales may come from the kernel launched just before this one
  griddep_wait();

  // With RS, registers move from warpgroup 0 (one TMA thread, one MMA thread) to
  // the epilogue warpgroups; the host launches this form only when the shares add
  // up to the block's registers.
  if (warp < L::FIRST_EPI) {
  if constexpr (RS) setmaxnreg_dec<L::REG_LO>();
  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int64_t issued = 0;
      for (int t = blockIdx.x; t < p.tiles && !*abort_flag; t += gridDim.x) {
        int mb, nb;
        tile_coords(p, t, mb, nb);
        for (int kb = 0; kb < p.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
          mbar_arrive_expect_tx(&full[stage], L::A_BYTES + L::B_BYTES);
          tma_load_2d(&tmA, &full[stage], smem + L::OFF_A + stage * L::A_BYTES, kb * BK, mb * BM);
          tma_load_2d(&tmB, &full[stage], smem + L::OFF_B + stage * L::B_BYTES, kb * BK, nb * BN);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      const int outstanding = static_cast<int>(issued < STAGES ? issued : STAGES);
      for (int j = 1; j <= outstanding; ++j) {
        int s = static_cast<int>(stage) - j;
        uint32_t ph = phase;
        if (s < 0) {
          s += STAGES;
          ph ^= 1u;
        }
        volatile int never = 0;
        mbar_wait(&full[s], ph, &never, p.status, kWaitTimeoutNs);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0 && DET) {
      // deterministic fold: each K range of the split accumulates into its own buffer
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      uint32_t stage = 0, phase = 0, acc_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        for (int r = 0; ok && r < p.det_splits; ++r) {
          const int b0 = det_kb_begin(r, p.num_kb, p.det_splits), b1 = det_kb_begin(r + 1, p.num_kb, p.det_splits);
          const uint32_t acc = acc_i % NACC;
          ok = mbar_wait(&tempty[acc], ((acc_i / NACC) & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          for (int kb = b0; kb < b1; ++kb) {
            ok = mbar_wait(&full[stage], phase, abort_flag, p.status, p.timeout_ns);
            if (!ok) break;
            tc_fence_after();
            const uint32_t d = tmem_base + acc * BN;
            const uint64_t adesc = smem_desc_sw128(smem_u32(smem + L::OFF_A + stage * L::A_BYTES));
            const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + L::OFF_B + stage * L::B_BYTES));
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k)
              mma_f8f6f4(d, adesc + static_cast<uint64_t>(k * UMMA_K / 16),
                         bdesc + static_cast<uint64_t>(k * UMMA_K / 16), idesc, (kb > b0 || k != 0) ? 1u : 0u);
            mma_commit(&empty[stage]);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(&tfull[acc]);
          ++acc_i;
        }
      }
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, p.status, kWaitTimeoutNs);
    } else if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      uint32_t stage = 0, phase = 0, acc_i = 0;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < p.tiles; t += gridDim.x) {
        for (int kb = 0; ok && kb < p.num_kb; ++kb) {
          const uint32_t acc = acc_i % NACC;
          ok = mbar_wait(&tempty[acc], ((acc_i / NACC) & 1u) ^ 1u, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          ok = mbar_wait(&full[stage], phase, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          const uint32_t d = tmem_base + acc * BN;
          const uint64_t adesc = smem_desc_sw128(smem_u32(smem + L::OFF_A + stage * L::A_BYTES));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(smem + L::OFF_B + stage * L::B_BYTES));
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            mma_f8f6f4(d, adesc + static_cast<uint64_t>(k * UMMA_K / 16),
                       bdesc + static_cast<uint64_t>(k * UMMA_K / 16), idesc, k != 0 ? 1u : 0u);
          mma_commit(&empty[stage]);
          mma_commit(&tfull[acc]);
          ++acc_i;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, p.status, kWaitTimeoutNs);
    }
  }
  } else {
    if constexpr (RS) setmaxnreg_inc<L::REG_HI>();
    // ------------------------------------------------------------- epilogue
    const int ew = warp - L::FIRST_EPI;
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int h = ew >> 2;                    // column slice
    uint8_t* stage_buf = smem + L::OFF_D + ew * 2 * L::D_BYTES;
    int dbuf = 0;
    uint32_t acc_i = 0;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + h * HALF;
    bool ok = true;
    for (int t = blockIdx.x; DET && ok && t < p.tiles; t += gridDim.x) {
      // deterministic fold: acc = p_0, then acc += p_r in range order, then the
      // row scale, column scale and bias by det_out
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int r0 = mb * BM + q * 32;
      const int nbase = nb * BN;
      float accum[HALF];
      for (int r = 0; ok && r < p.det_splits; ++r) {
        const uint32_t acc = acc_i % NACC;
        ok = mbar_wait(&tfull[acc], (acc_i / NACC) & 1u, abort_flag, p.status, p.timeout_ns);
        if (!ok) break;
        tc_fence_after();
        // two 32-column loads in flight: chunk c + 1 is requested before chunk c is added
        uint32_t rv[2][32];
        tmem_ld_32x32b_x32(lane_addr + acc * BN, rv[0]);
#pragma unroll
        for (int c = 0; c < HALF / 32; ++c) {
          tmem_ld_wait();
          if (c + 1 < HALF / 32) tmem_ld_32x32b_x32(lane_addr + acc * BN + (c + 1) * 32, rv[(c + 1) & 1]);
          if (c + 1 == HALF / 32) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            accum[c * 32 + j] =
                r == 0 ? __uint_as_float(rv[c & 1][j]) : __fadd_rn(accum[c * 32 + j], __uint_as_float(rv[c & 1][j]));
        }
        ++acc_i;
      }
      if (!ok) break;
      const float sa = a_scale_at(p, row);
      const float sb_t = p.b_mode == 0 ? __ldg(p.b_scale) : 1.0f;
#pragma unroll
      for (int c = 0; c < HALF / 32; ++c) {
        const int n0 = nbase + h * HALF + c * 32;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = n0 + 2 * j;   // N is a multiple of 8, so n < N covers n + 1
          float s0 = sb_t, s1 = sb_t, b0 = 0.0f, b1 = 0.0f;
          if (n < p.N) {
            if (p.b_mode == 1) {
              s0 = __ldg(p.b_scale + n);
              s1 = __ldg(p.b_scale + n + 1);
            }
            if (p.bias) {
              b0 = __bfloat162float(p.bias[n]);
              b1 = __bfloat162float(p.bias[n + 1]);
            }
          }
          w[j] = pack2(det_out(accum[c * 32 + 2 * j], sa, s0, b0), det_out(accum[c * 32 + 2 * j + 1], sa, s1, b1),
                       p.out_fp16);
        }
        if (store_block(&tmD, stage_buf + dbuf * L::D_BYTES, w, lane, n0, r0, p.M, p.N)) dbuf ^= 1;
      }
    }
    for (int t = blockIdx.x; !DET && ok && t < p.tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int row = mb * BM + q * 32 + lane;
      const int r0 = mb * BM + q * 32;
      const int nbase = nb * BN;
      float accum[HALF];
#pragma unroll
      for (int j = 0; j < HALF; ++j) accum[j] = 0.0f;
      const ScaleStream<AMODE, BBLOCK> ss(p, row, nbase + h * HALF);
      // K blocks in groups of four: the scale words of the next group are loaded while
      // this one is folded (a packed UE8M0 word holds all four A scales of a group)
      constexpr bool PACKED = AMODE == FP8MM_SCALE_A_GROUP128_UE8M0;
      uint32_t na[4];
      float nbw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        na[u] = (PACKED && u > 0) ? 0u : ss.a_raw(u);
        nbw[u] = ss.b_raw(u);
      }
      for (int kg = 0; kg < p.num_kb && ok; kg += 4) {
        uint32_t ca[4];
        float cb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ca[u] = na[u];
          cb[u] = nbw[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          na[u] = (PACKED && u > 0) ? 0u : ss.a_raw(kg + 4 + u);
          nbw[u] = ss.b_raw(kg + 4 + u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int kb = kg + u;
          if (kb >= p.num_kb) break;
          const uint32_t acc = acc_i % NACC;
          ok = mbar_wait(&tfull[acc], (acc_i / NACC) & 1u, abort_flag, p.status, p.timeout_ns);
          if (!ok) break;
          tc_fence_after();
          const float sk = ScaleStream<AMODE, BBLOCK>::decode(ca[PACKED ? 0 : u], kb) * cb[u];
          // kFoldCols-column chunks; the buffer goes back to the MMA warp once its last
          // chunk is in registers
#pragma unroll
          for (int c = 0; c < HALF / kFoldCols; ++c) {
            uint32_t rv[kFoldCols];
            if constexpr (kFoldCols == 64)
              tmem_ld_32x32b_x64(lane_addr + acc * BN + c * 64, *reinterpret_cast<uint32_t(*)[64]>(rv));
            else
              tmem_ld_32x32b_x32(lane_addr + acc * BN + c * 32, *reinterpret_cast<uint32_t(*)[32]>(rv));
            tmem_ld_wait();
            if (c + 1 == HALF / kFoldCols) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[acc]);
            }
#pragma unroll
            for (int j = 0; j < kFoldCols; ++j)
              accum[c * kFoldCols + j] = fmaf(sk, __uint_as_float(rv[j]), accum[c * kFoldCols + j]);
          }
          ++acc_i;
        }
      }
      if (!ok) break;
      // column scale (per tensor or per column; block scales were applied per K block)
      // and bias, two columns at a time (N is a multiple of 8, so n < N covers n + 1)
      const float sb_t = p.b_mode == 0 ? __ldg(p.b_scale) : 1.0f;
#pragma unroll
      for (int c = 0; c < HALF / 32; ++c) {
        const int n0 = nbase + h * HALF + c * 32;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const int n = n0 + 2 * j;
          float s0 = sb_t, s1 = sb_t, b0 = 0.0f, b1 = 0.0f;
          if (n < p.N) {
            if (p.b_mode == 1) {
              s0 = __ldg(p.b_scale + n);
              s1 = __ldg(p.b_scale + n + 1);
            }
            if (p.bias) {
              b0 = __bfloat162float(p.bias[n]);
              b1 = __bfloat162float(p.bias[n + 1]);
            }
          }
          const float a0 = accum[c * 32 + 2 * j], a1 = accum[c * 32 + 2 * j + 1];
          w[j] = pack2(a0 * s0 + b0, a1 * s1 + b1, p.out_fp16);
        }
        if (store_block(&tmD, stage_buf + dbuf * L::D_BYTES, w, lane, n0, r0, p.M, p.N)) dbuf ^= 1;
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------------------ small-M: swap-AB + split-K
//
// For few rows (M <= 128) the weight is what has to stream from HBM, and a
// 128 x BN tile grid has far fewer tiles than SMs.  Here the MMA's 128-row
// operand is a 128-row slice of the weight B and the N = BT operand is the
// token block of A, so D^T[n, m] accumulates in TMEM (lane = n, column = m).
// The K range of a tile is split across the S CTAs of a thread-block cluster;
// each CTA writes its fp32 partial [BT][128] into its own shared memory
// (reusing the drained stage ring), and after a cluster barrier CTA r sums
// rows [r*128/S, (r+1)*128/S) of all S partials in rank order 0..S-1 through
// distributed shared memory, scales, rounds and stores them.  One launch, no
// global workspace, and a fixed summation order.

template <int BT>
struct SwapLayout {
  static constexpr int W_BYTES = 128 * BK;          // weight slice per stage
  static constexpr int X_BYTES = BT * BK;           // token block per stage
  static constexpr int STAGES = BT <= 32 ? 5 : (BT == 64 ? 4 : 3);
  static constexpr int RING = STAGES * (W_BYTES + X_BYTES);
  static constexpr int PART = BT * 128 * 4;         // fp32 partial, aliases the ring
  static constexpr int DATA = RING > PART ? RING : PART;
  static constexpr int OFF_BAR = DATA;
  static constexpr int NBARS = 2 * STAGES + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int OFF_VEC = (OFF_MISC + 16 + 15) / 16 * 16;   // b_scale[128], bias[128], a_scale[BT]
  static constexpr int ALLOC = OFF_VEC + (256 + BT) * 4 + 1024;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(BT);
  static_assert(X_BYTES % 1024 == 0, "token block must keep 1024-byte alignment");
};

struct SplitArgs {
  int splits;     // cluster size S
  int n_tiles;    // ceil(N / 128)
};

// The split-K reduction of the swap-AB kernel: thread t of the 128 epilogue threads
// takes outputs idx = t, t + 128, ... of this rank's share (idx -> token m = idx /
// quads, rows r_begin + 4 (idx % quads) .. + 3), sums the S partials of each in rank
// order 0..S-1 through distributed shared memory, scales, adds the bias and stores.
// U outputs per pass, all U x S loads issued before the first sum (S <= SMAX): with
// two outputs a pass, large token blocks were bound by the remote-load round trips.
struct SwapReduce {
  uint32_t part_addr;
  int t, total, quads, r_begin, S, m0, n0;
  const float* vec_sa;
  const float* vec_sb;
  const float* vec_bias;

  template <int U, int SMAX>
  __device__ __forceinline__ void run(const GemmArgs& p, __nv_bfloat16* out) const {
    for (int base = t; base < total; base += 128 * U) {
      float4 pv[U][SMAX];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * 128;
        const int m = idx < total ? idx / quads : 0;
        const int row = idx < total ? r_begin + 4 * (idx - m * quads) : r_begin;
        const uint32_t off = static_cast<uint32_t>((m * 128 + row) * 4);
#pragma unroll
        for (int s2 = 0; s2 < SMAX; ++s2)
          if (s2 < S && (U == 2 || idx < total))   // wide passes skip loads past the share
            pv[u][s2] = ld_dsmem_f32x4(mapa_shared(part_addr + off, static_cast<uint32_t>(s2)));
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * 128;
        if (idx >= total) break;
        float4 acc = pv[u][0];
#pragma unroll
        for (int s2 = 1; s2 < SMAX; ++s2) {
          if (s2 < S) {
            acc.x += pv[u][s2].x;
            acc.y += pv[u][s2].y;
            acc.z += pv[u][s2].z;
            acc.w += pv[u][s2].w;
          }
        }
        const int m = idx / quads;
        const int row = r_begin + 4 * (idx - m * quads);
        const int n = n0 + row;
        if (n >= p.N) continue;
        const float sa = vec_sa[m];
        const float4 sb = *reinterpret_cast<const float4*>(vec_sb + row);
        const float4 bs = *reinterpret_cast<const float4*>(vec_bias + row);
        const float v0 = acc.x * sa * sb.x + bs.x, v1 = acc.y * sa * sb.y + bs.y;
        const float v2 = acc.z * sa * sb.z + bs.z, v3 = acc.w * sa * sb.w + bs.w;
        const int64_t o = static_cast<int64_t>(m0 + m) * p.N + n;
        *reinterpret_cast<uint2*>(out + o) = make_uint2(pack2(v0, v1, p.out_fp16), pack2(v2, v3, p.out_fp16));
      }
    }
  }
};

template <int BT>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_swap_splitk_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                                const GemmArgs p, const SplitArgs sp, __nv_bfloat16* out) {
  // A kernel launched after this one on the stream as a programmatic dependent (the
  // next GEMM of a decode step) may start its set-up and its weight prefetch now; it
  // reads what this kernel writes only after griddepcontrol.wait
  griddep_launch_dependents();
  using L = SwapLayout<BT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + L::STAGES;
  uint64_t* tfull = empty + L::STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  float* vec_sb = reinterpret_cast<float*>(smem + L::OFF_VEC);
  float* vec_bias = vec_sb + 128;
  float* vec_sa = vec_bias + 128;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = sp.splits;
  const int rank = static_cast<int>(cluster_ctarank());
  const int n_tile = blockIdx.x / S;
  const int m0 = blockIdx.y * BT;
  const int n0 = n_tile * 128;
  const int kb0 = static_cast<int>(static_cast<int64_t>(rank) * p.num_kb / S);
  const int kb1 = static_cast<int>(static_cast<int64_t>(rank + 1) * p.num_kb / S);

  // The first ring's worth of loads is issued by the producer thread right after the
  // barriers exist, before TMEM allocation and the block barrier.
  const int pre = kb1 - kb0 < L::STAGES ? kb1 - kb0 : L::STAGES;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmW);
    tma_prefetch_desc(&tmX);
    for (int s = 0; s < L::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // while the kernel launched before this one finishes, pull the first ring's weight
    // slices into L2; every load into shared memory waits for that kernel (it may have
    // written the weight as well as the tokens)
    for (int j = 0; j < pre; ++j) tma_prefetch_l2_2d(&tmW, (kb0 + j) * BK, n0);
    griddep_wait();
    for (int j = 0; j < pre; ++j) {
      mbar_arrive_expect_tx(&full[j], L::W_BYTES + L::X_BYTES);
      uint8_t* st = smem + j * (L::W_BYTES + L::X_BYTES);
      tma_load_2d(&tmW, &full[j], st, (kb0 + j) * BK, n0);
      tma_load_2d(&tmX, &full[j], st + L::W_BYTES, (kb0 + j) * BK, m0);
    }
  }

  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();   // A and its scales may come from the kernel launched just before
  float* part = reinterpret_cast<float*>(smem);   // [BT][128], valid after the mainloop

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = pre % L::STAGES, phase = pre == L::STAGES ? 1u : 0u;
      int issued = pre;
      for (int kb = kb0 + pre; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&full[stage], L::W_BYTES + L::X_BYTES);
        uint8_t* st = smem + stage * (L::W_BYTES + L::X_BYTES);
        tma_load_2d(&tmW, &full[stage], st, kb * BK, n0);
        tma_load_2d(&tmX, &full[stage], st + L::W_BYTES, kb * BK, m0);
        ++issued;
        if (++stage == L::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      const int outstanding = issued < L::STAGES ? issued : L::STAGES;
      for (int j = 1; j <= outstanding; ++j) {
        int s = static_cast<int>(stage) - j;
        uint32_t ph = phase;
        if (s < 0) {
          s += L::STAGES;
          ph ^= 1u;
        }
        volatile int never = 0;
        mbar_wait(&full[s], ph, &never, p.status, kWaitTimeoutNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(128, BT);
      uint32_t stage = 0, phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status, p.timeout_ns)) break;
        tc_fence_after();
        uint8_t* st = smem + stage * (L::W_BYTES + L::X_BYTES);
        const uint64_t adesc = smem_desc_sw128(smem_u32(st));
        const uint64_t bdesc = smem_desc_sw128(smem_u32(st + L::W_BYTES));
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k)
          mma_f8f6f4(tmem_base, adesc + static_cast<uint64_t>(k * UMMA_K / 16),
                     bdesc + static_cast<uint64_t>(k * UMMA_K / 16), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[stage]);
        if (++stage == L::STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit(tfull);
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, p.status, kWaitTimeoutNs);
    }
  } else {
    {
      // the epilogue's column scales, bias and row scales, fetched while the weights stream
      const int t = threadIdx.x - 64;
      const int n = n0 + t;
      vec_sb[t] = n < p.N ? (p.b_mode == 0 ? __ldg(p.b_scale) : __ldg(p.b_scale + n)) : 0.0f;
      vec_bias[t] = (p.bias && n < p.N) ? __bfloat162float(p.bias[n]) : 0.0f;
      for (int m = t; m < BT; m += 128) vec_sa[m] = a_scale_at(p, m0 + m);
    }
    // TMEM -> own shared-memory partial [BT][128] (lane = weight row within the tile)
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (mbar_wait(tfull, 0, abort_flag, p.status, p.timeout_ns)) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < BT / 16; ++c) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 16, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) part[(c * 16 + j) * 128 + row] = __uint_as_float(r[j]);
      }
    }
    tc_fence_before();
  }

  __syncwarp();
  cluster_sync_all();   // every partial of the cluster is in shared memory

  if (warp >= 2) {
    // rank r sums rows [r * rows_per, ...) of the tile, four consecutive rows per thread
    const int t = threadIdx.x - 64;
    const int rows_per = ((128 + S - 1) / S + 3) & ~3;
    const int r_begin = rank * rows_per;
    const int r_count = max(0, min(rows_per, 128 - r_begin));
    const int quads = r_count >> 2;
    const int mt = min(BT, p.M - m0);
    const int total = quads * mt;
    const uint32_t part_addr = smem_u32(part);
    // a CTA of the cluster that gave up left stale data in its partial (the status word
    // holds the error): then no CTA of the cluster writes the tile
    bool no_abort = true;
    for (int s2 = 0; s2 < S; ++s2)
      no_abort &= ld_dsmem_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), static_cast<uint32_t>(s2))) == 0;
    // two outputs per thread per pass for 16- and 32-token blocks (decode: one pass);
    // 64- and 128-token blocks keep about 16 remote loads in flight per thread
    if (no_abort) {
      const SwapReduce r{part_addr, t, total, quads, r_begin, S, m0, n0, vec_sa, vec_sb, vec_bias};
      if constexpr (BT >= 64) {
        if (S <= 2)
          r.run<8, 2>(p, out);
        else if (S <= 4)
          r.run<4, 4>(p, out);
        else
          r.run<2, 8>(p, out);
      } else {
        r.run<2, 8>(p, out);
      }
    }
  }

  __syncwarp();
  cluster_sync_all();   // no CTA leaves while others may still read its partial
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ------------------------------------- deterministic split, small M: cluster
//
// The batch-invariant mode splits K into S ranges fixed by N and K (never by M).  For
// few rows the S CTAs of a cluster each accumulate one range of a 128 x BN tile in
// TMEM (the same instruction shape and K order as the fold kernel), copy the valid
// rows of their fp32 partial into shared memory (over the drained ring), and after a
// cluster barrier CTA r sums its share of the tile's outputs over the S partials in
// range order through distributed shared memory -- ((p_0 + p_1) + p_2) ... exactly as
// the fold kernel adds its range accumulators -- and applies det_out.

template <int BN, int STAGES>
struct DetLayout {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int RING = STAGES * (A_BYTES + B_BYTES);
  static constexpr int PSTRIDE = BN + 4;             // floats per partial row (conflict-free v4 stores)
  static constexpr int PART = BM * PSTRIDE * 4;
  static constexpr int DATA = RING > PART ? RING : PART;
  static constexpr int OFF_BAR = DATA;
  static constexpr int NBARS = 2 * STAGES + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int ALLOC = OFF_MISC + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = pow2_at_least(BN);
  static_assert((A_BYTES + B_BYTES) % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    fp8_gemm_det_cluster_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                                const GemmArgs p, void* out) {
  griddep_launch_dependents();   // as in the small-M kernel
  using L = DetLayout<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* drain = tfull + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.det_splits;
  const int rank = static_cast<int>(cluster_ctarank());
  const int n0 = (blockIdx.x / S) * BN;
  const int m0 = blockIdx.y * BM;
  const int rows = min(BM, p.M - m0);                 // valid rows of this tile
  const int kb0 = det_kb_begin(rank, p.num_kb, S), kb1 = det_kb_begin(rank + 1, p.num_kb, S);
  constexpr int STAGE_BYTES = L::A_BYTES + L::B_BYTES;

  // the first ring's worth of loads goes out as soon as the barriers exist
  const int pre = kb1 - kb0 < STAGES ? kb1 - kb0 : STAGES;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the first ring's weight tiles into L2 while the kernel before this one finishes;
    // the loads themselves wait for it
    for (int j = 0; j < pre; ++j) tma_prefetch_l2_2d(&tmB, (kb0 + j) * BK, n0);
    griddep_wait();
    for (int j = 0; j < pre; ++j) {
      mbar_arrive_expect_tx(&full[j], STAGE_BYTES);
      uint8_t* st = smem + j * STAGE_BYTES;
      tma_load_2d(&tmA, &full[j], st, (kb0 + j) * BK, m0);
      tma_load_2d(&tmB, &full[j], st + L::A_BYTES, (kb0 + j) * BK, n0);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();
  float* part = reinterpret_cast<float*>(smem);       // [rows][PSTRIDE], valid after the mainloop

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = pre % STAGES, phase = pre == STAGES ? 1u : 0u;
      int issued = pre;
      for (int kb = kb0 + pre; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status, p.timeout_ns)) break;
        mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
        uint8_t* st = smem + stage * STAGE_BYTES;
        tma_load_2d(&tmA, &full[stage], st, kb * BK, m0);
        tma_load_2d(&tmB, &full[stage], st + L::A_BYTES, kb * BK, n0);
        ++issued;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      const int outstanding = issued < STAGES ? issued : STAGES;
      for (int j = 1; j <= outstanding; ++j) {
        int s = static_cast<int>(stage) - j;
        uint32_t ph = phase;
        if (s < 0) {
          s += STAGES;
          ph ^= 1u;
        }
        volatile int never = 0;
        mbar_wait(&full[s], ph, &never, p.status, kWaitTimeoutNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
      uint32_t stage = 0, phase = 0;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&full[stage], phase, abort_flag, p.status, p.timeout_ns)) break;
        tc_fence_after();
        uint8_t* st = smem + stage * STAGE_BYTES;
        const uint64_t adesc = smem_desc_sw128(smem_u32(st));
        const uint64_t bdesc = smem_desc_sw128(smem_u32(st + L::A_BYTES));
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k)
          mma_f8f6f4(tmem_base, adesc + static_cast<uint64_t>(k * UMMA_K / 16),
                     bdesc + static_cast<uint64_t>(k * UMMA_K / 16), idesc, (kb > kb0 || k > 0) ? 1u : 0u);
        mma_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      mma_commit(tfull);
      mma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, p.status, kWaitTimeoutNs);
    }
  } else {
    // TMEM -> own partial: lane = row within the tile; the valid rows only
    const int q = warp & 3;
    const int row = q * 32 + lane;
    if (q * 32 < rows && mbar_wait(tfull, 0, abort_flag, p.status, p.timeout_ns)) {
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + c * 32, r);
        tmem_ld_wait();
        if (row < rows) {
          float4* dst = reinterpret_cast<float4*>(part + row * L::PSTRIDE + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
        }
      }
    }
    tc_fence_before();
  }

  __syncwarp();
  cluster_sync_all();   // every partial of the cluster is in shared memory, every abort flag final

  // a CTA that gave up left stale data in its partial: then no CTA of the cluster
  // writes the tile (the status word already holds the error)
  bool any_abort = false;
  for (int s2 = 0; s2 < S; ++s2)
    any_abort |= ld_dsmem_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), static_cast<uint32_t>(s2))) != 0;

  if (!any_abort) {
    // CTA rank takes outputs [i0, i1) of the tile's rows x BN/4 column quads
    constexpr int QUADS = BN / 4;
    const int items = rows * QUADS;
    const int i0 = static_cast<int>(static_cast<int64_t>(rank) * items / S);
    const int i1 = static_cast<int>(static_cast<int64_t>(rank + 1) * items / S);
    const uint32_t part_addr = smem_u32(part);
    for (int i = i0 + static_cast<int>(threadIdx.x); i < i1; i += kThreads) {
      const int row = i / QUADS;
      const int col = (i - row * QUADS) * 4;
      const int n = n0 + col;
      if (n >= p.N) continue;     // N is a multiple of 8: a quad is wholly in or out
      const uint32_t off = static_cast<uint32_t>((row * L::PSTRIDE + col) * 4);
      float4 acc = ld_dsmem_f32x4(mapa_shared(part_addr + off, 0));
      for (int s2 = 1; s2 < S; ++s2) {
        const float4 v = ld_dsmem_f32x4(mapa_shared(part_addr + off, static_cast<uint32_t>(s2)));
        acc.x = __fadd_rn(acc.x, v.x);
        acc.y = __fadd_rn(acc.y, v.y);
        acc.z = __fadd_rn(acc.z, v.z);
        acc.w = __fadd_rn(acc.w, v.w);
      }
      const float sa = a_scale_at(p, m0 + row);
      float sb[4], bs[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sb[j] = p.b_mode == 0 ? __ldg(p.b_scale) : __ldg(p.b_scale + n + j);
        bs[j] = p.bias ? __bfloat162float(p.bias[n + j]) : 0.0f;
      }
      const uint32_t lo = pack2(det_out(acc.x, sa, sb[0], bs[0]), det_out(acc.y, sa, sb[1], bs[1]), p.out_fp16);
      const uint32_t hi = pack2(det_out(acc.z, sa, sb[2], bs[2]), det_out(acc.w, sa, sb[3], bs[3]), p.out_fp16);
      *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + static_cast<int64_t>(m0 + row) * p.N + n) =
          make_uint2(lo, hi);
    }
  }

  __syncwarp();
  cluster_sync_all();   // no CTA leaves while others may still read its partial
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

struct Config {
  int bn, stages;
  bool group_a;
};

template <int BN, int STAGES>
cudaError_t launch(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const GemmArgs& p,
                   int grid, cudaStream_t st) {
  using L = Layout<BN, STAGES>;
  auto kern = fp8_gemm_kernel<BN, STAGES>;
  const cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), L::ALLOC);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(grid), dim3(kThreads), L::ALLOC, st, 0, ta, tb, td, p);
}

// Group-scale tiles: 128 x 256 with two accumulators and a register split (the
// preferred form), or 128 x 192 without one.  The split is used only if the kernel
// was built with the register count its setmaxnreg shares assume.
constexpr int kGroupBN = 256;
constexpr int kGroupBNAlt = 192;

template <int AMODE, bool BBLOCK>
struct GroupKernels {
  using LS = GroupLayout<kGroupBN, 4, 2, 2, true>;
  using LA = GroupLayout<kGroupBNAlt, 4, 2, 3, false>;
  static constexpr auto split = fp8_gemm_group_kernel<kGroupBN, 4, 2, 2, true, AMODE, BBLOCK>;
  static constexpr auto alt = fp8_gemm_group_kernel<kGroupBNAlt, 4, 2, 3, false, AMODE, BBLOCK>;

  // Once per device: shared-memory opt-in for both, and whether the split kernel's
  // register count covers its setmaxnreg shares (otherwise its warps would wait).
  static cudaError_t prepare(bool* split_ok) {
    const int r = once_per_device(reinterpret_cast<const void*>(split), []() {
      cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, LS::ALLOC);
      if (e == cudaSuccess) e = cudaFuncSetAttribute(alt, cudaFuncAttributeMaxDynamicSharedMemorySize, LA::ALLOC);
      cudaFuncAttributes fa;
      if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, split);
      if (e != cudaSuccess) return -static_cast<int>(e);
      return 128 * LS::REG_LO + 32 * LS::EPI_WARPS * LS::REG_HI <= LS::THREADS * fa.numRegs ? 1 : 0;
    });
    if (r < 0) return static_cast<cudaError_t>(-r);
    *split_ok = r == 1;
    return cudaSuccess;
  }

  static cudaError_t launch(bool use_split, const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                            const GemmArgs& p, int grid, cudaStream_t st) {
    if (use_split) return launch_pdl(split, dim3(grid), dim3(LS::THREADS), LS::ALLOC, st, 0, ta, tb, td, p);
    return launch_pdl(alt, dim3(grid), dim3(LA::THREADS), LA::ALLOC, st, 0, ta, tb, td, p);
  }
};

// The runtime scale modes mapped onto the compiled specialisations.
#define FP8MM_GROUP_DISPATCH(a_mode, bblock, CALL)                                              \
  do {                                                                                          \
    if (bblock) {                                                                               \
      if ((a_mode) == FP8MM_SCALE_A_GROUP128) return GroupKernels<FP8MM_SCALE_A_GROUP128, true>::CALL; \
      if ((a_mode) == FP8MM_SCALE_A_GROUP128_COLMAJOR)                                          \
        return GroupKernels<FP8MM_SCALE_A_GROUP128_COLMAJOR, true>::CALL;                       \
      return GroupKernels<FP8MM_SCALE_A_GROUP128_UE8M0, true>::CALL;                            \
    }                                                                                           \
    if ((a_mode) == FP8MM_SCALE_A_GROUP128) return GroupKernels<FP8MM_SCALE_A_GROUP128, false>::CALL; \
    if ((a_mode) == FP8MM_SCALE_A_GROUP128_COLMAJOR)                                            \
      return GroupKernels<FP8MM_SCALE_A_GROUP128_COLMAJOR, false>::CALL;                        \
    return GroupKernels<FP8MM_SCALE_A_GROUP128_UE8M0, false>::CALL;                             \
  } while (0)

cudaError_t group_prepare(int a_mode, bool bblock, bool* split_ok) {
  FP8MM_GROUP_DISPATCH(a_mode, bblock, prepare(split_ok));
}

cudaError_t group_launch(int a_mode, bool bblock, bool use_split, const CUtensorMap& ta, const CUtensorMap& tb,
                         const CUtensorMap& td, const GemmArgs& p, int grid, cudaStream_t st) {
  FP8MM_GROUP_DISPATCH(a_mode, bblock, launch(use_split, ta, tb, td, p, grid, st));
}
#undef FP8MM_GROUP_DISPATCH

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

template <int BT>
cudaError_t launch_swap(const CUtensorMap& tw, const CUtensorMap& tx, const GemmArgs& p, int splits, void* out,
                        cudaStream_t st) {
  using L = SwapLayout<BT>;
  auto kern = fp8_gemm_swap_splitk_kernel<BT>;
  const cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), L::ALLOC);
  if (e != cudaSuccess) return e;
  SplitArgs sp;
  sp.splits = splits;
  sp.n_tiles = ceil_div(p.N, 128);
  return launch_pdl(kern, dim3(static_cast<unsigned>(sp.n_tiles * splits), static_cast<unsigned>(ceil_div(p.M, BT)), 1),
                    dim3(kThreads), L::ALLOC, st, static_cast<unsigned>(splits), tw, tx, p, sp,
                    static_cast<__nv_bfloat16*>(out));
}

// Split count for the small-M path: as many K slices (cluster size <= 8, at least two
// K blocks each) as keep every CTA resident at two CTAs per SM, and no more than keep
// the fp32 partials (S x token block x 128 x 4 bytes, written then read) under half
// the weight bytes of a tile -- under all of them for 128-token blocks, whose CTAs
// stream as many token bytes as weight bytes, so that more K slices shorten both
// (measured at M = 128, K = 4096: four slices instead of two take N = 4096 from 18.8
// to 16.5 us; 64-token blocks lose with eight slices instead of four).
int pick_splits(int64_t M, int64_t N, int num_kb, int sms) {
  const int64_t tiles = static_cast<int64_t>(ceil_div(N, 128)) * ceil_div(M, 128);
  int s = 1;
  const int64_t bt = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
  const int64_t cap = static_cast<int64_t>(num_kb) * BK / ((bt == 128 ? 8 : 16) * bt);
  while (s < 8 && s + 1 <= cap && tiles * (s + 1) <= 2LL * sms && (s + 1) * 2 <= num_kb) ++s;
  return s;
}

// ----------------------------------------------- deterministic split: host side

// Tile width of the deterministic mode, from N alone.
int det_bn(int64_t N) { return N >= 1024 ? 256 : (N >= 256 ? 128 : 64); }

// K ranges of the deterministic mode, from N and K alone: enough ranges that a small-M
// problem spreads its weight stream over about kDetTargetCtas CTAs, at most eight
// (the cluster size) and at least two K blocks each.  A fixed target, not the
// device's SM count: the split must not depend on anything but N and K.  The target
// trades the two ends: every range adds a fold to each tile of a large problem
// (about 2 % of its time each at K = 4096), while too few leave a small problem's
// weight stream on too few SMs; measured on K = 4096, N = 4096, a target of 64
// (four ranges) costs 1.02-1.17x the normal launch at M <= 16 and 1.2x at M = 4096,
// 152 (eight ranges, clusters of eight 197 KB CTAs) 1.5x and 1.45x.
constexpr int kDetTargetCtas = 64;
int det_splits(int64_t N, int num_kb) {
  const int64_t n_tiles = (N + det_bn(N) - 1) / det_bn(N);
  int64_t s = kDetTargetCtas / n_tiles;
  s = s < 8 ? s : 8;
  s = s < num_kb / 2 ? s : num_kb / 2;
  return s < 1 ? 1 : static_cast<int>(s);
}

template <int BN, int STAGES>
cudaError_t launch_det_cluster(const CUtensorMap& ta, const CUtensorMap& tb, const GemmArgs& p, void* out,
                               cudaStream_t st) {
  using L = DetLayout<BN, STAGES>;
  auto kern = fp8_gemm_det_cluster_kernel<BN, STAGES>;
  const cudaError_t e = smem_opt_in(reinterpret_cast<const void*>(kern), L::ALLOC);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(static_cast<unsigned>(p.n_blocks * p.det_splits), static_cast<unsigned>(p.m_blocks), 1),
                    dim3(kThreads), L::ALLOC, st, static_cast<unsigned>(p.det_splits), ta, tb, p, out);
}

// The fold form of the deterministic split for each tile width: 128 x 256 with the
// register split of the group kernel (eight epilogue warps), 128 x 128 and 128 x 64
// with four.
template <int BN> struct DetFold;
template <> struct DetFold<256> {
  using L = GroupLayout<256, 4, 2, 2, true>;
  static constexpr auto kern = fp8_gemm_group_kernel<256, 4, 2, 2, true, kAModeDetFold, false>;
};
template <> struct DetFold<128> {
  using L = GroupLayout<128, 6, 2, 1, false>;
  static constexpr auto kern = fp8_gemm_group_kernel<128, 6, 2, 1, false, kAModeDetFold, false>;
};
template <> struct DetFold<64> {
  using L = GroupLayout<64, 8, 2, 1, false>;
  static constexpr auto kern = fp8_gemm_group_kernel<64, 8, 2, 1, false, kAModeDetFold, false>;
};

// Once per device: shared-memory opt-in, and whether the fold kernel may run (with a
// register split, only if the compiled register count covers its shares).  Returns 1
// if it may, 0 if not, or a negative CUDA error.
template <int BN>
int det_fold_prepare() {
  using F = DetFold<BN>;
  return once_per_device(reinterpret_cast<const void*>(F::kern), []() {
    cudaError_t e = cudaFuncSetAttribute(F::kern, cudaFuncAttributeMaxDynamicSharedMemorySize, F::L::ALLOC);
    cudaFuncAttributes fa;
    if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, F::kern);
    if (e != cudaSuccess) return -static_cast<int>(e);
    if (!F::L::FIRST_EPI || F::L::FIRST_EPI == 2) return 1;   // no register split
    return 128 * F::L::REG_LO + 32 * F::L::EPI_WARPS * F::L::REG_HI <= F::L::THREADS * fa.numRegs ? 1 : 0;
  });
}

template <int BN>
cudaError_t launch_det_fold(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td, const GemmArgs& p,
                            int grid, cudaStream_t st) {
  using F = DetFold<BN>;
  return launch_pdl(F::kern, dim3(grid), dim3(F::L::THREADS), F::L::ALLOC, st, 0, ta, tb, td, p);
}

// Shape-keyed tile table.  Deterministic mode picks its tile from N alone, so every M
// (and every prefix / suffix of the rows) runs the same tile, K order and instruction;
// otherwise the width with the smallest estimated time wins.
Config pick_config(int64_t M, int64_t N, bool deterministic, bool group_a, int sms) {
  if (group_a) return {kGroupBN, 4, true};
  if (deterministic) {
    if (N >= 1024) return {256, 4, false};
    if (N >= 256) return {128, 6, false};
    return {64, 8, false};
  }
  // Estimated time ~ waves x tile width / relative MMA efficiency of that width
  // (measured on the prefill shapes: BN = 128 runs at 0.6 of BN = 256's rate; BN = 64
  // lower still), so a partly idle single wave of wide tiles can beat two waves of
  // narrow ones.
  const int64_t mblk = ceil_div(M, BM);
  // relative MMA rate of a 128 x N instruction stream, 3N / (512 + N): a fixed cost
  // per K step plus one proportional to N, fitted to the measured 0.6 at N = 128
  constexpr int kOpts = 5;
  const Config opts[kOpts] = {{256, 4, false}, {224, 4, false}, {192, 5, false}, {128, 6, false}, {64, 8, false}};
  int best = 0;
  double best_cost = 0.0;
  for (int i = 0; i < kOpts; ++i) {
    const double eff = 3.0 * opts[i].bn / (512.0 + opts[i].bn);
    const int64_t tiles = mblk * ceil_div(N, opts[i].bn);
    const double cost = static_cast<double>((tiles + sms - 1) / sms) * opts[i].bn / eff;
    if (i == 0 || cost < best_cost) {
      best = i;
      best_cost = cost;
    }
  }
  return opts[best];
}

}  // namespace
}  // namespace fp8mm

using namespace fp8mm;

extern "C" int fp8_scaled_mm(const void* A, const void* B, const float* a_scale, const float* b_scale, int scale_mode,
                             const void* bias, void* out, int out_dtype, int64_t M, int64_t N, int64_t K, int64_t lda,
                             int64_t ldb, int deterministic, fp8mm_stream_t stream) {
  const int a_mode = scale_mode & 0xF;
  const int b_mode = (scale_mode >> 4) & 0xF;
  if (M < 0 || N < 0) return FP8MM_EINVAL;
  if (a_mode > FP8MM_SCALE_A_GROUP128_UE8M0 || b_mode > 2 || (scale_mode & ~0xFF)) return FP8MM_EINVAL;
  if (b_mode == 2 && a_mode < FP8MM_SCALE_A_GROUP128) return FP8MM_EINVAL;   // block B goes with group A
  if (out_dtype != FP8MM_DTYPE_BF16 && out_dtype != FP8MM_DTYPE_FP16) return FP8MM_EINVAL;
  if (M > 0x7fffffff || N > 0x7fffffff || K > 0x7fffffff) return FP8MM_EINVAL;
  if (K <= 0 || K % 16 != 0 || lda < K || ldb < K) return FP8MM_EINVAL;
  if (lda % 16 != 0 || ldb % 16 != 0 || N % 8 != 0) return FP8MM_EALIGN;
  const bool group_a = a_mode >= FP8MM_SCALE_A_GROUP128;
  if (group_a && K % 128 != 0) return FP8MM_EINVAL;
  if (M == 0 || N == 0) return FP8MM_OK;
  if (!A || !B || !a_scale || !b_scale || !out) return FP8MM_EINVAL;
  if (!aligned16(A) || !aligned16(B) || !aligned16(out)) return FP8MM_EALIGN;
  if ((reinterpret_cast<uintptr_t>(a_scale) & 3u) || (reinterpret_cast<uintptr_t>(b_scale) & 3u) ||
      (reinterpret_cast<uintptr_t>(bias) & 1u))
    return FP8MM_EALIGN;
  {
    // out must not overlap the inputs
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(out), o1 = o0 + static_cast<uintptr_t>(M * N * 2);
    auto overlaps = [&](const void* p, int64_t bytes) {
      const uintptr_t b0 = reinterpret_cast<uintptr_t>(p);
      return p && b0 < o1 && o0 < b0 + static_cast<uintptr_t>(bytes);
    };
    if (overlaps(A, (M - 1) * lda + K) || overlaps(B, (N - 1) * ldb + K) || overlaps(bias, N * 2))
      return FP8MM_EINVAL;
  }
  int* status = status_word_device_ptr();
  const int sms = num_sms();
  if (!status || sms <= 0) return FP8MM_ECUDA;

  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs p;
  p.M = static_cast<int>(M);
  p.N = static_cast<int>(N);
  p.K = static_cast<int>(K);
  p.num_kb = ceil_div(K, BK);
  p.a_mode = a_mode;
  p.b_mode = b_mode;
  p.a_ld = a_mode == FP8MM_SCALE_A_GROUP128 ? K / 128 : (M + 3) / 4 * 4;
  p.b_ld = K / 128;
  p.a_scale = a_scale;
  p.b_scale = b_scale;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.out_fp16 = out_dtype == FP8MM_DTYPE_FP16;
  p.det_splits = 1;
  p.status = status;
  p.timeout_ns = wait_timeout_ns();

  if (deterministic && !group_a) {
    // batch-invariant split: the tile width from N, the K ranges from N and K; the
    // cluster kernel when the whole problem fits in one wave of clusters, else the
    // persistent fold kernel -- the same bits either way
    const int bn = det_bn(N);
    p.det_splits = det_splits(N, p.num_kb);
    p.m_blocks = ceil_div(M, BM);
    p.n_blocks = ceil_div(N, bn);
    p.tiles = p.m_blocks * p.n_blocks;
    const int fold_ok = bn == 256 ? det_fold_prepare<256>() : (bn == 128 ? det_fold_prepare<128>() : det_fold_prepare<64>());
    if (fold_ok < 0) return FP8MM_ECUDA;
    CUtensorMap ta, tb, td;
    if (!make_tma_2d(&ta, const_cast<void*>(A), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, BK, BM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tma_2d(&tb, const_cast<void*>(B), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, BK, bn,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tma_2d(&td, out, out_dtype == FP8MM_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     N, M, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
      return FP8MM_ECUDA;
    cudaError_t e;
    if (fold_ok == 0 || static_cast<int64_t>(p.tiles) * p.det_splits <= sms) {
      if (bn == 256)
        e = launch_det_cluster<256, 4>(ta, tb, p, out, st);
      else if (bn == 128)
        e = launch_det_cluster<128, 6>(ta, tb, p, out, st);
      else
        e = launch_det_cluster<64, 8>(ta, tb, p, out, st);
    } else {
      p.raster = 8;
      const int grid = p.tiles < sms ? p.tiles : sms;
      if (bn == 256)
        e = launch_det_fold<256>(ta, tb, td, p, grid, st);
      else if (bn == 128)
        e = launch_det_fold<128>(ta, tb, td, p, grid, st);
      else
        e = launch_det_fold<64>(ta, tb, td, p, grid, st);
    }
    return e == cudaSuccess ? FP8MM_OK : FP8MM_ECUDA;
  }

  if (!group_a && M <= 128) {
    // small M: swap-AB with split-K over a cluster
    const int bt = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
    const int splits = pick_splits(M, N, p.num_kb, sms);
    CUtensorMap tw, tx;
    if (!make_tma_2d(&tw, const_cast<void*>(B), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, BK, 128,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tma_2d(&tx, const_cast<void*>(A), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, BK, bt,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return FP8MM_ECUDA;
    p.m_blocks = ceil_div(M, bt);
    p.n_blocks = ceil_div(N, 128);
    p.tiles = p.m_blocks * p.n_blocks;
    p.raster = 1;
    cudaError_t e;
    switch (bt) {
      case 16: e = launch_swap<16>(tw, tx, p, splits, out, st); break;
      case 32: e = launch_swap<32>(tw, tx, p, splits, out, st); break;
      case 64: e = launch_swap<64>(tw, tx, p, splits, out, st); break;
      default: e = launch_swap<128>(tw, tx, p, splits, out, st); break;
    }
    return e == cudaSuccess ? FP8MM_OK : FP8MM_ECUDA;
  }

  Config cfg = pick_config(M, N, deterministic != 0, group_a, sms);
  bool group_split = false;
  if (group_a) {
    const cudaError_t e = group_prepare(a_mode, b_mode == 2, &group_split);
    if (e != cudaSuccess) return FP8MM_ECUDA;
    if (!group_split) cfg.bn = kGroupBNAlt;
  }
  CUtensorMap ta, tb, td;
  if (!make_tma_2d(&ta, const_cast<void*>(A), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, BK, BM,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tma_2d(&tb, const_cast<void*>(B), CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, BK, cfg.bn,
                   CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tma_2d(&td, out, out_dtype == FP8MM_DTYPE_FP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                           : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                   N, M, N * 2, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return FP8MM_ECUDA;

  p.m_blocks = ceil_div(M, BM);
  p.n_blocks = ceil_div(N, cfg.bn);
  p.tiles = p.m_blocks * p.n_blocks;
  // Raster group: as many M blocks as keep the group's A panel (rows x K bytes) within
  // about 48 MB of the 126 MB L2, so the panel is re-read from L2, not HBM, while the
  // group sweeps N, and B is fetched from HBM once per group.
  {
    int64_t fit = (48ll << 20) / (static_cast<int64_t>(BM) * K);
    fit = fit < 8 ? 8 : fit;
    const int64_t groups = (p.m_blocks + fit - 1) / fit;            // then balance the groups
    p.raster = static_cast<int>((p.m_blocks + groups - 1) / groups);
  }
  const int grid = p.tiles < sms ? p.tiles : sms;
  cudaError_t e;
  if (cfg.group_a)
    e = group_launch(a_mode, b_mode == 2, group_split, ta, tb, td, p, grid, st);
  else if (cfg.bn == 256)
    e = launch<256, 4>(ta, tb, td, p, grid, st);
  else if (cfg.bn == 224)
    e = launch<224, 4>(ta, tb, td, p, grid, st);
  else if (cfg.bn == 192)
    e = launch<192, 5>(ta, tb, td, p, grid, st);
  else if (cfg.bn == 128)
    e = launch<128, 6>(ta, tb, td, p, grid, st);
  else
    e = launch<64, 8>(ta, tb, td, p, grid, st);
  return e == cudaSuccess ? FP8MM_OK : FP8MM_ECUDA;
}
