// Backward GEMMs of the routed/shared SwiGLU experts on CTA pairs (tcgen05
// cta_group::2, sm_103a), with MN-major shared-memory operands where the
// contraction runs along a tensor's rows.
//
// Rows live in the padded slot space: every group (expert) starts at a
// multiple of 64 rows and its pad rows hold zeros in x_pad and dy_pad, so a
// K loop over a group's rows needs no masking (zero rows add nothing).
//
//   kBwdDH    dh = dy . W_down[e]            token rows x H   (K = d)
//             A = dy_pad (K-major), B = W_down [E][d][H] read MN-major;
//             epilogue: dA = [dh * u * SiLU'(a) | dh * SiLU(a)] from the
//             recomputed pre-activations AU = [a | u] (bf16).
//   kBwdDX    dz = dA . W_gu[e]              token rows x d   (K = 2H)
//             A = dA_pad (K-major), B = W_gu [E][2H][d] read MN-major; fp32 out.
//   kBwdDWD   dW_down[e] = dy^T . h          d x H            (K = rows of e)
//             A = dy_pad read MN-major, B = h_pad read MN-major; fp32 out.
//   kBwdDWGU  dW_gu[e] = dA^T . x            2H x d           (K = rows of e)
//             A = dA_pad read MN-major, B = x_pad read MN-major; fp32 out.
//
// An MN-major tile is staged as 64-wide boxes of 64 K rows (128-byte
// swizzle): the MMA descriptor's leading-byte offset is the stride between
// 64-wide boxes (8 KB), the stride-byte offset the stride between 8-row K
// groups (1 KB), and a K step of 16 advances the start by 2 KB.
//
// Pair tile: M = 256 (128 rows per CTA), N = 256 or 128 (N/2 rows of B per
// CTA).  Warp roles, the barrier protocol, bounded waits and the abort path
// follow the forward pair kernel (gemm_tc.cu).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace bw {

constexpr int BK = 64;
constexpr int A_BYTES = 128 * BK * 2;  // 16 KB
constexpr int B_BYTES = 128 * BK * 2;  // 16 KB (N = 256); N = 128 uses half
// A ring stage holds KSUB consecutive K blocks (each A then B, 32 KB): the MMA issuer waits
// once and commits once per stage.
constexpr int KSUB = 2;
constexpr int SUB_BYTES = A_BYTES + B_BYTES;
constexpr int STAGE_BYTES = KSUB * SUB_BYTES;
constexpr int STAGES = 6 / KSUB;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
// per epilogue warp: 32 x 33 fp32 (gradient chunks) or two 32 x 40 bf16 tiles (kBwdDH)
// (the fp32 path's full quarters use the first 4 KB as a {32, 32} TMA store box)
constexpr int EPI_STAGE_FLOATS = 32 * 40;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 3072 + 4 * EPI_STAGE_FLOATS * 4;
constexpr int PAIR_GROUP = 8;

struct Shared {  // must stay below 3072 bytes: the epilogue staging tiles follow it
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  int gmb[257];  // token-row modes: first m-tile of each group; weight modes: unused
  int gpb[257];  // token-row modes: first pair of each group
};

static_assert(sizeof(Shared) <= 3072, "control block overlaps the epilogue staging tiles");
static_assert(2 * 32 * 40 * 2 <= EPI_STAGE_FLOATS * 4 && 32 * 33 <= EPI_STAGE_FLOATS,
              "epilogue staging tiles exceed a warp's area");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory above the per-CTA limit");
static_assert(32 * 32 * 4 <= EPI_STAGE_FLOATS * 4 && (EPI_STAGE_FLOATS * 4) % 1024 == 0 &&
                  (STAGES * STAGE_BYTES + 3072) % 1024 == 0,
              "each warp's staging area holds a 1024-byte-aligned {32, 32} fp32 TMA box");

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Shared* sh,
                                         unsigned* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (sh->abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        sh->abort_flag = 1;
        record_status(status, MOE_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Shared-memory matrix descriptor, 128-byte swizzle; K-major (lbo unused, 16) or
// MN-major (lbo = stride between 64-wide boxes).
__device__ __forceinline__ uint64_t desc(uint32_t addr, uint32_t lbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>(1024u >> 4) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(2u) << 61;
  return d;
}

constexpr bool a_mn(int mode) { return mode == kBwdDWD || mode == kBwdDWGU; }
// kBwdDH and kBwdDWD tile the hidden units (H per weight slice, a multiple of 128): N = 256,
// and 128 for the last tile of a slice when H is an odd multiple of 128.
constexpr bool n_tiles_hidden(int mode) { return mode == kBwdDH || mode == kBwdDWD; }

struct Tile {
  int group;   // expert / shared slice
  int m0;      // token modes: first token row of this CTA's m-tile; weight modes: first output row of this CTA
  int nrows;   // token modes: valid rows of this CTA's m-tile (0 for an empty peer half)
  int n0;      // first output column of the pair tile
  int ncols;   // output columns of the pair tile (MMA N): 256, or 128 at the end of a slice
  int sl;      // kBwdDH: weight slice of the tile (shared experts), 0 routed
  int h_in;    // kBwdDH: first hidden unit of the tile inside its slice
  int k_rows;  // weight modes: first token row of the group (K origin)
  int n_kb;    // K blocks
};

// Pair tile -> this CTA's work.  Token modes walk (group, blocks of PAIR_GROUP
// pairs of m-tiles, N tiles with the pairs fastest) like the forward kernel;
// weight modes walk (group, output-row tile, output-column tile).
template <int MODE>
__device__ __forceinline__ Tile tile_info(const BwdArgs& a, const Shared* sh, int tile,
                                          uint32_t rank) {
  Tile t;
  if (!a_mn(MODE)) {
    const int NT = a.n_ntiles;
    int lo = 0, hi = a.n_groups;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (sh->gpb[mid] * NT <= tile) lo = mid; else hi = mid;
    }
    const int beg = sh->gpb[lo], cnt = sh->gpb[lo + 1] - beg;
    const int local = tile - beg * NT;
    const int blk = local / (PAIR_GROUP * NT);
    const int within = local - blk * PAIR_GROUP * NT;
    const int bs = min(PAIR_GROUP, cnt - blk * PAIR_GROUP);
    const int nt = within / bs;
    const int pi = blk * PAIR_GROUP + (within - nt * bs);
    const int m_in_group = 2 * pi + static_cast<int>(rank);
    const int4 lead = a.mt_info[sh->gmb[lo] + 2 * pi];
    t.group = lead.x;
    if (m_in_group < sh->gmb[lo + 1] - sh->gmb[lo]) {
      const int4 m = a.mt_info[sh->gmb[lo] + m_in_group];
      t.m0 = m.y;
      t.nrows = m.z;
    } else {
      t.m0 = lead.y + lead.z;
      t.nrows = 0;
    }
    if (MODE == kBwdDH) {
      t.sl = nt / a.nt_per_slice;
      t.h_in = (nt - t.sl * a.nt_per_slice) * 256;
      t.ncols = min(256, a.n_per_slice - t.h_in);
      t.n0 = t.sl * a.n_per_slice + t.h_in;
    } else {
      t.sl = 0;
      t.h_in = 0;
      t.ncols = 256;
      t.n0 = nt * 256;
    }
    t.k_rows = 0;
    t.n_kb = a.n_kblocks;
  } else {
    const int per_group = a.n_mtiles * a.n_ntiles;
    t.group = tile / per_group;
    const int local = tile - t.group * per_group;
    const int mt = local / a.n_ntiles;
    const int nt = local - mt * a.n_ntiles;
    t.m0 = mt * 256 + static_cast<int>(rank) * 128;
    t.nrows = 128;
    t.n0 = nt * 256;
    t.ncols = n_tiles_hidden(MODE) ? min(256, a.n_cols - t.n0) : 256;
    t.sl = 0;
    t.h_in = 0;
    if (a.group_rows) {
      t.k_rows = a.group_rows[t.group];
      t.n_kb = (a.group_rows[t.group + 1] - t.k_rows) / BK;
    } else {
      t.k_rows = 0;
      t.n_kb = a.rows_shared / BK;
    }
  }
  return t;
}

template <int MODE>
__device__ __forceinline__ int total_tiles(const BwdArgs& a, const Shared* sh) {
  if (!a_mn(MODE)) return sh->gpb[a.n_groups] * a.n_ntiles;
  return a.n_groups * a.n_mtiles * a.n_ntiles;
}

// This CTA's loads of K block kb (both CTAs complete on the leader's `full`).
template <int MODE>
__device__ __forceinline__ void issue_kblock(const BwdArgs& a, const CUtensorMap* tmA,
                                             const CUtensorMap* tmB, const Tile& t, int kb,
                                             uint32_t rank, uint32_t full, uint32_t sa,
                                             uint32_t sb) {
  const int r = static_cast<int>(rank);
  if (MODE == kBwdDH) {
    // A: dy rows, K = d.  B: W_down[slice] rows f (K) x columns h (N): ncols/2 h per CTA
    // as 64-wide boxes.
    const int h0 = t.h_in + r * (t.ncols / 2);
    ptx::tma_load_2d_pair(sa, tmA, full, kb * BK, t.m0);
    for (int b = 0; b < t.ncols / 128; ++b)
      ptx::tma_load_3d_pair(sb + b * 8192, tmB, full, h0 + 64 * b, kb * BK, t.group + t.sl);
  } else if (MODE == kBwdDX) {
    // A: dA rows, K = 2H (spanning slices for the shared experts).  B: W_gu[slice]
    // rows j (K) x columns c (N), 128 c per CTA as two 64-wide boxes.
    const int kslice = kb / a.kb_per_slice;
    const int kin = (kb - kslice * a.kb_per_slice) * BK;
    const int c0 = t.n0 + r * 128;
    ptx::tma_load_2d_pair(sa, tmA, full, kb * BK, t.m0);
    ptx::tma_load_3d_pair(sb, tmB, full, c0, kin, t.group + kslice);
    ptx::tma_load_3d_pair(sb + 8192, tmB, full, c0 + 64, kin, t.group + kslice);
  } else if (MODE == kBwdDWD) {
    // A: dy^T: rows f of this CTA (two 64-wide boxes), K = the group's token rows.
    // B: h^T: 64 columns h per CTA.
    const int krow = t.k_rows + kb * BK;
    const int hcol = a.b_col0 + t.group * a.b_col_stride + t.n0 + r * (t.ncols / 2);
    ptx::tma_load_2d_pair(sa, tmA, full, t.m0, krow);
    ptx::tma_load_2d_pair(sa + 8192, tmA, full, t.m0 + 64, krow);
    for (int b = 0; b < t.ncols / 128; ++b)
      ptx::tma_load_2d_pair(sb + b * 8192, tmB, full, hcol + 64 * b, krow);
  } else {  // kBwdDWGU
    const int krow = t.k_rows + kb * BK;
    const int jcol = t.group * a.a_col_stride + t.m0;
    const int c0 = t.n0 + r * 128;
    ptx::tma_load_2d_pair(sa, tmA, full, jcol, krow);
    ptx::tma_load_2d_pair(sa + 8192, tmA, full, jcol + 64, krow);
    ptx::tma_load_2d_pair(sb, tmB, full, c0, krow);
    ptx::tma_load_2d_pair(sb + 8192, tmB, full, c0 + 64, krow);
  }
}

// logistic sigmoid with the approximate divide (its error is far below the bf16 rounding of dA)
__device__ __forceinline__ float sigm(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 p = __bfloat1622float2(h[i]);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
  }
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Epilogue for output row `r` (TMEM lane) of this CTA, columns col0.. of the accumulator.
// `stage`: this warp's EPI_STAGE_FLOATS-float staging area in shared memory.
template <int MODE>
__device__ __forceinline__ void epilogue(const BwdArgs& a, const Tile& t, uint32_t col0, int r,
                                         float* stage, const CUtensorMap* tmO) {
  const int NCOL = t.ncols;
  if (MODE == kBwdDH) {
    // dh for hidden units [n0, n0 + 128) of this warp's 32 rows; AU = [a | u] per slice.
    // Per 32-column chunk the warp brings a and u of its 32 rows into shared memory with
    // 4 lanes per row (64 contiguous bytes each), every thread turns its row into
    // [da | du] in place, and the warp writes them back the same way.
    const int lane = r & 31;
    const int row_w = r - lane;
    const int rows_here = min(32, t.nrows - row_w);
    const long long col_a = static_cast<long long>(t.sl) * 2 * a.n_per_slice + t.h_in;
    const long long row0 = static_cast<long long>(t.m0) + row_w;
    // two 32 x 32 bf16 tiles (a, u) with rows padded to 40 elements (80 bytes: 16-byte
    // aligned rows; the 4-lane row accesses of a quarter-warp hit distinct banks)
    __nv_bfloat16* ta = reinterpret_cast<__nv_bfloat16*>(stage);
    __nv_bfloat16* tu = ta + 32 * 40;
    const int lr = lane >> 2, lseg = lane & 3;  // cooperative access: row lr + 8 i, 16-byte segment lseg
    // [a, u] of the next chunk are loaded into registers while the current one is
    // computed, so a chunk's global loads overlap the previous chunk's work.
    uint4 na[4], nu[4];
    auto load_au = [&](int c) {
      const long long col = col_a + c * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = lr + 8 * i;
        na[i] = nu[i] = make_uint4(0, 0, 0, 0);
        if (rr < rows_here) {
          const __nv_bfloat16* src = a.au + (row0 + rr) * a.ld_au + col + lseg * 8;
          na[i] = *reinterpret_cast<const uint4*>(src);
          nu[i] = *reinterpret_cast<const uint4*>(src + a.n_per_slice);
        }
      }
    };
    load_au(0);
#pragma unroll 1
    for (int c = 0; c < NCOL / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
      ptx::tmem_ld_wait();
      const long long col = col_a + c * 32;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = lr + 8 * i;
        *reinterpret_cast<uint4*>(ta + rr * 40 + lseg * 8) = na[i];
        *reinterpret_cast<uint4*>(tu + rr * 40 + lseg * 8) = nu[i];
      }
      if (c + 1 < NCOL / 32) load_au(c + 1);
      __syncwarp();
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float av[8], uv[8];
        unpack8(*reinterpret_cast<const uint4*>(ta + lane * 40 + q * 8), av);
        unpack8(*reinterpret_cast<const uint4*>(tu + lane * 40 + q * 8), uv);
        uint32_t pa[4], pu[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float da2[2], du2[2];
#pragma unroll
          for (int z = 0; z < 2; ++z) {
            const int e = 2 * i + z;
            const float dh = __uint_as_float(v[q * 8 + e]);
            const float sg = sigm(av[e]);
            da2[z] = dh * uv[e] * (sg * (1.0f + av[e] * (1.0f - sg)));
            du2[z] = dh * av[e] * sg;
          }
          pa[i] = pack2(da2[0], da2[1]);
          pu[i] = pack2(du2[0], du2[1]);
        }
        *reinterpret_cast<uint4*>(ta + lane * 40 + q * 8) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
        *reinterpret_cast<uint4*>(tu + lane * 40 + q * 8) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
      }
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rr = lr + 8 * i;
        if (rr < rows_here) {
          __nv_bfloat16* dst = a.out_bf16 + (row0 + rr) * a.ld_out + col + lseg * 8;
          *reinterpret_cast<uint4*>(dst) = *reinterpret_cast<const uint4*>(ta + rr * 40 + lseg * 8);
          *reinterpret_cast<uint4*>(dst + a.n_per_slice) =
              *reinterpret_cast<const uint4*>(tu + rr * 40 + lseg * 8);
        }
      }
      __syncwarp();
    }
  } else {
    const int lane = r & 31;
    const int row_w = r - lane;  // first row of this warp's quarter
    const int rows_here = min(32, t.nrows - row_w);  // valid rows of this warp's quarter
    // a group without rows (no K blocks) has a zero gradient, not the stale accumulator
    const bool zero = t.n_kb == 0;
    if (rows_here == 32) {
      // fp32 output of a full quarter: each 32 x 32 chunk is written to shared memory in
      // the 128-byte-swizzled layout of a {32, 32} TMA box (thread = row, eight 16-byte
      // stores to distinct banks per quarter-warp) and stored by one TMA bulk store
      const int orow = MODE == kBwdDX
                           ? t.m0 + row_w
                           : static_cast<int>(t.group * a.out_group_rows) + t.m0 + row_w;
      uint8_t* my_row = reinterpret_cast<uint8_t*>(stage) + lane * 128;
      const uint32_t src = ptx::smem_u32(stage);
#pragma unroll 1
      for (int c = 0; c < NCOL / 32; ++c) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
        ptx::tmem_ld_wait();
        if (c > 0) {
          if (lane == 0) ptx::bulk_wait_read0();  // the previous chunk's store has read the box
          __syncwarp();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 q = zero ? make_uint4(0, 0, 0, 0)
                               : make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          *reinterpret_cast<uint4*>(my_row + ((j ^ (lane & 7)) << 4)) = q;
        }
        ptx::fence_proxy_async_smem_cta();
        __syncwarp();
        if (lane == 0) {
          ptx::tma_store_2d(tmO, src, t.n0 + c * 32, orow);
          ptx::bulk_commit();
        }
      }
      if (lane == 0) ptx::bulk_wait_read0();  // the box is free for the next tile
      __syncwarp();
      return;
    }
    // a partial quarter: each 32-row x 32-column chunk goes through a padded shared-memory
    // tile, so every store instruction writes one row's 128 contiguous bytes
    float* obase;
    if (MODE == kBwdDX)
      obase = a.out_f32 + (static_cast<long long>(t.m0) + row_w) * a.ld_out + t.n0;
    else
      obase = a.out_f32 + static_cast<long long>(t.group) * a.out_group_stride +
              (static_cast<long long>(t.m0) + row_w) * a.ld_out + t.n0;
#pragma unroll 1
    for (int c = 0; c < NCOL / 32; ++c) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) stage[lane * 33 + i] = zero ? 0.f : __uint_as_float(v[i]);
      __syncwarp();
      for (int i = 0; i < rows_here; ++i)
        obase[static_cast<long long>(i) * a.ld_out + c * 32 + lane] = stage[i * 33 + lane];
      __syncwarp();
    }
  }
}

}  // namespace bw

template <int MODE>
__global__ void __launch_bounds__(bw::NUM_THREADS, 1)
    bwd_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmO, const BwdArgs args) {
  using namespace bw;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t smem0 = ptx::smem_u32(smem);
  // bytes both CTAs load per stage: A 16 KB each, B ncols/2 rows each

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sh->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sh->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&sh->tmem_full[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&sh->tmem_empty[a]), 8);
    }
    ptx::mbar_init(ptx::smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (MODE != kBwdDH) ptx::prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&sh->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  pdl_wait();
  if (!a_mn(MODE)) {
    for (int g = threadIdx.x; g <= args.n_groups; g += blockDim.x)
      sh->gmb[g] = args.group_mt_begin[g];
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int g = 0; g < args.n_groups; ++g) {
        sh->gpb[g] = run;
        run += (sh->gmb[g + 1] - sh->gmb[g] + 1) >> 1;
      }
      sh->gpb[args.n_groups] = run;
    }
  }
  __syncthreads();
  const uint32_t tmem_base = sh->tmem_base;
  const int n_tiles = total_tiles<MODE>(args, sh);
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cluster; tile < n_tiles && ok; tile += n_clusters) {
      const Tile t = tile_info<MODE>(args, sh, tile, rank);
      const uint32_t TX = 2u * static_cast<uint32_t>(A_BYTES + (t.ncols / 2) * BK * 2);
      for (int kb0 = 0; kb0 < t.n_kb; kb0 += KSUB) {
        const int nsub = min(KSUB, t.n_kb - kb0);
        if (!wait_bar(ptx::smem_u32(&sh->empty[stage]), phase ^ 1u, sh, args.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = ptx::smem_u32(&sh->full[stage]) & ptx::kLeaderMask;
          if (rank == 0) ptx::mbar_arrive_expect_tx(full, static_cast<uint32_t>(nsub) * TX);
          for (int u = 0; u < nsub; ++u) {
            const uint32_t sa = smem0 + stage * STAGE_BYTES + u * SUB_BYTES;
            bw::issue_kblock<MODE>(args, &tmA, &tmB, t, kb0 + u, rank, full, sa, sa + A_BYTES);
          }
        }
        __syncwarp();
        if (++stage == STAGES) stage = 0, phase ^= 1u;
      }
    }
    if (!ok) {
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (rank == 0) {
      const uint32_t idesc_flags = (static_cast<uint32_t>(a_mn(MODE)) << 15) | (1u << 16);
      const uint32_t a_lbo = a_mn(MODE) ? 8192u : 16u;
      const uint32_t a_step = a_mn(MODE) ? (2048u >> 4) : (32u >> 4);
      const uint32_t b_step = 2048u >> 4;
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = cluster; tile < n_tiles && ok; tile += n_clusters, ++local) {
        const Tile t = tile_info<MODE>(args, sh, tile, rank);
        const uint32_t idesc = ptx::idesc_bf16_f32(256, t.ncols) | idesc_flags;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!wait_bar(ptx::smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1u, sh, args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * 256;
        for (int kb0 = 0; kb0 < t.n_kb; kb0 += KSUB) {
          const int nsub = min(KSUB, t.n_kb - kb0);
          if (!wait_bar(ptx::smem_u32(&sh->full[stage]), phase, sh, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          if (lane == 0) {
            for (int u = 0; u < nsub; ++u) {
              const uint32_t sa = smem0 + stage * STAGE_BYTES + u * SUB_BYTES;
              const uint64_t adesc = bw::desc(sa, a_lbo);
              const uint64_t bdesc = bw::desc(sa + A_BYTES, 8192u);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                ptx::umma_bf16_pair(d_tmem, adesc + a_step * kk, bdesc + b_step * kk, idesc,
                                    (kb0 + u > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::umma_commit_pair(ptx::smem_u32(&sh->empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
        if (!ok) break;
        if (lane == 0) ptx::umma_commit_pair(ptx::smem_u32(&sh->tmem_full[acc]), 0x3);
        __syncwarp();
      }
      if (!ok) {
        if (lane == 0) ptx::umma_commit_pair_local(ptx::smem_u32(&sh->drain));
        __syncwarp();
        const uint64_t t0 = globaltimer_ns();
        while (!ptx::mbar_try_wait(ptx::smem_u32(&sh->drain), 0) &&
               globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5, both CTAs)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    // after the control block (Shared, < 3 KB): 4 x EPI_STAGE_FLOATS floats, inside SMEM_BYTES
    float* epi_stage = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 3072) +
                       (warp - 2) * EPI_STAGE_FLOATS;
    int local = 0;
    for (int tile = cluster; tile < n_tiles; tile += n_clusters, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      if (!wait_bar(ptx::smem_u32(&sh->tmem_full[acc]), acc_phase, sh, args.status)) break;
      ptx::tc_fence_after();
      const Tile t = tile_info<MODE>(args, sh, tile, rank);
      bw::epilogue<MODE>(args, t, lane_addr + acc * 256, r, epi_stage, &tmO);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t e = ptx::smem_u32(&sh->tmem_empty[acc]);
        if (rank == 0) ptx::mbar_arrive(e);
        else ptx::mbar_arrive_cluster(ptx::mapa(e, 0));
      }
    }
    if (MODE != kBwdDH && lane == 0) ptx::bulk_wait0();  // this warp's TMA stores are performed
    __syncwarp();
  }

  pdl_trigger();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  // looked up once (a function-local static is initialised once, even with concurrent callers)
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return nullptr;
  }();
  return fn;
}

// bf16 tensor map, 128-byte swizzle, box {64, box_rows[, 1]} over [outer][rows][inner].
bool make_map(CUtensorMap* m, int rank, const void* base, uint64_t inner, uint64_t rows,
              uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 output [rows][inner] for TMA stores of {32, 32} boxes, 128-byte swizzle
bool make_out_map(CUtensorMap* m, float* base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 4};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE>
cudaError_t launch(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo,
                   const BwdArgs& args, int num_sms, cudaStream_t stream) {
  static OncePerDevice<64> once;
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const cudaError_t set_up = once.run(dev, [&]() -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(bwd_gemm_pair_kernel<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         bw::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t q = {};
    cudaLaunchAttribute ca;
    ca.id = cudaLaunchAttributeClusterDimension;
    ca.val.clusterDim.x = 2;
    ca.val.clusterDim.y = 1;
    ca.val.clusterDim.z = 1;
    q.gridDim = dim3(2 * (num_sms / 2));
    q.blockDim = dim3(bw::NUM_THREADS);
    q.dynamicSmemBytes = bw::SMEM_BYTES;
    q.attrs = &ca;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, bwd_gemm_pair_kernel<MODE>, &q) != cudaSuccess || n <= 0)
      n = num_sms / 2;
    if (dev < 64) max_clusters[dev] = n;
    return cudaSuccess;
  });
  if (set_up != cudaSuccess) return set_up;
  int clusters = num_sms / 2;
  if (dev < 64 && max_clusters[dev] < clusters) clusters = max_clusters[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(bw::NUM_THREADS);
  cfg.dynamicSmemBytes = bw::SMEM_BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = 2;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, bwd_gemm_pair_kernel<MODE>, ma, mb, mo, args);
}

}  // namespace

cudaError_t bwd_gemm(int mode, const BwdGemmOperands& op, const BwdArgs& args_in, int num_sms,
                     cudaStream_t stream) {
  CUtensorMap ma, mb, mo;
  BwdArgs args = args_in;
  switch (mode) {
    case kBwdDH:
      // A: dy_pad [rows][K]; B: W_down [slices][K = d][N = H] read MN-major (box 64 x 64)
      if (!make_map(&ma, 2, op.A, op.a_inner, op.a_rows, 1, 128) ||
          !make_map(&mb, 3, op.B, op.b_inner, op.b_rows, op.b_slices, 64))
        return cudaErrorInvalidValue;
      return launch<kBwdDH>(ma, mb, ma, args, num_sms, stream);
    case kBwdDX:
      // output dz [rows of A][ld_out]
      if (!make_map(&ma, 2, op.A, op.a_inner, op.a_rows, 1, 128) ||
          !make_map(&mb, 3, op.B, op.b_inner, op.b_rows, op.b_slices, 64) ||
          !make_out_map(&mo, args.out_f32, args.ld_out, op.a_rows))
        return cudaErrorInvalidValue;
      return launch<kBwdDX>(ma, mb, mo, args, num_sms, stream);
    case kBwdDWD:
    case kBwdDWGU: {
      // output: n_groups gradients of out_group_stride elements, rows of ld_out
      if (args.ld_out <= 0 || args.out_group_stride % args.ld_out != 0) return cudaErrorInvalidValue;
      args.out_group_rows = args.out_group_stride / args.ld_out;
      if (!make_map(&ma, 2, op.A, op.a_inner, op.a_rows, 1, 64) ||
          !make_map(&mb, 2, op.B, op.b_inner, op.b_rows, 1, 64) ||
          !make_out_map(&mo, args.out_f32, args.ld_out, args.out_group_rows * args.n_groups))
        return cudaErrorInvalidValue;
      return mode == kBwdDWD ? launch<kBwdDWD>(ma, mb, mo, args, num_sms, stream)
                             : launch<kBwdDWGU>(ma, mb, mo, args, num_sms, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
