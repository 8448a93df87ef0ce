// Persistent grouped GEMM on tcgen05 tensor cores (sm_103a), bf16 in, fp32
// accumulate in TMEM, for the routed-expert FFN and the condensation
// similarity tiles.
//
//   D[m, n] = sum_k A[row0 + m, k] * B[slice, n0 + n, k]     (both operands K-major)
//
// One CTA per SM.  Warp 0 issues TMA loads into a shared-memory ring, warp 1
// allocates TMEM and has one thread issue tcgen05.mma into one of two 256-column
// fp32 accumulators, warps 2-5 drain the other accumulator through tcgen05.ld and
// run the epilogue, so the epilogue of tile i overlaps the main loop of tile i+1.
// The expert FFN (kSwiGLU, kStore) and the similarity tiles (kSimBits) run on CTA
// pairs (cta_group::2, M=256 x N=256, below); the router logits (kRouter) on single
// CTAs (M=128, a 4-stage ring).
//
// Epilogues:
//   kSwiGLU  B rows are loaded as 128 gate rows then 128 up rows of the same
//            hidden units, so one accumulator holds gate|up; the epilogue writes
//            h = SiLU(gate) * up (bf16) -- the gate/up half of a SwiGLU expert.
//   kStore   writes D (bf16), optionally to a remapped output row.
//   kSimBits condensation (CTA pairs): D is a 256 x 256 tile of the bucket's Gram matrix;
//            the epilogue turns cos(x_i, x_j) >= tau, j < i, into bits.
//   kRouter  router logits: B is the fp32 router weight split exactly into
//            three bf16 terms.  With E up to 128 the terms sit side by side along N
//            (each E rounded up to 32 rows; one MMA up to 64 experts, two above -- terms
//            1 and 2, then term 3 -- into a 384-column accumulator): the K loop runs
//            over d, split across CTAs, and the epilogue adds the three accumulators;
//            otherwise the K loop runs over the three terms in turn (N = E rounded up
//            to 32).  The epilogue writes fp32 partial sums.
//
// Tiles.  Rows are grouped (one group per expert / bucket); a group's rows are
// cut into 128-row m-tiles (the last one ragged; rows past the group are
// computed but never stored).  For kSwiGLU/kStore the tile walk goes through the
// groups in order and, inside a group, through blocks of units (pairs of m-tiles)
// with the N tiles outside the units, so CTAs running at the same time share B
// tiles (weights) and A tiles (tokens) through L2 (the pair kernel's tile_info).
// kSimBits reads an explicit list of (pair of m-tiles, column tile).
//
// Every wait is bounded; on timeout the CTA records MOE_ERR_TIMEOUT, stops
// issuing work, drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace tc {

#ifdef MOE_FAULT_INJECTION
// Test build only: when set, the pair kernel's producers issue no TMA loads (the expected
// bytes never arrive), so the MMA warp's bounded wait on the full barrier runs out and the
// call ends with MOE_ERR_TIMEOUT in the device status word.
__device__ int g_fault_drop_loads = 0;
__device__ __forceinline__ bool fault_drop_loads() {
  return *reinterpret_cast<volatile int*>(&g_fault_drop_loads) != 0;
}
#else
__device__ __forceinline__ bool fault_drop_loads() { return false; }
#endif

constexpr int BM = 128, BN = 256, BK = 64;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;
constexpr int M_GROUP = 16;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align slack*/ + 2048 /*barriers, tables*/;
// the router's wide layout (65..128 experts): x's 16 KB and three 128-row terms per stage
constexpr int WIDE_STAGE_BYTES = A_BYTES + 3 * 128 * BK * 2;
constexpr int WIDE_STAGES = STAGES * STAGE_BYTES / WIDE_STAGE_BYTES;
static_assert(WIDE_STAGES * WIDE_STAGE_BYTES == STAGES * STAGE_BYTES, "one ring size");
static_assert(WIDE_STAGES <= STAGES && WIDE_STAGE_BYTES % 1024 == 0, "wide router stages");

enum Mode { kSwiGLU = 0, kStore = 1, kSimBits = 2, kRouter = 3 };

struct Shared {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  int gmb[257];  // group_mt_begin, staged once per CTA (tile lookups stay in shared memory)
};

// Bounded mbarrier wait.  Returns false if the CTA is aborting or the limit passed.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Shared* sh,
                                         unsigned* status) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = globaltimer_ns();
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

struct TileInfo {
  int slice;  // B slice (expert) of the m-tile
  int row0;   // first A row
  int nrows;  // valid rows (<= 128; a tail tile's up to kMaxTailRows)
  int gbase;  // first row of the group (bucket offset)
  int nt;     // N tile (or column tile for kSimBits)
  int tail = 0;  // CTA-pair kernel: 1 for a tail tile (weights as M, the m-tile's rows as N)
};

template <int MODE>
__device__ __forceinline__ TileInfo tile_info(const TcGemmArgs& a, const int* gmb, int tile) {
  int mt, nt;
  if (MODE == kRouter) {
    // one group of T rows; tile = (m-tile, K split), K splits fastest
    TileInfo t;
    const int m = tile / a.n_ntiles;
    t.nt = tile - m * a.n_ntiles;
    t.slice = 0;
    t.row0 = m * BM;
    t.nrows = min(BM, a.n_rows - t.row0);
    t.gbase = 0;
    return t;
  }
  {
    const int NT = a.n_ntiles;
    int lo = 0, hi = a.n_groups;  // largest g with begin[g] * NT <= tile
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (gmb[mid] * NT <= tile) lo = mid; else hi = mid;
    }
    const int beg = gmb[lo];
    const int cnt = gmb[lo + 1] - beg;
    const int local = tile - beg * NT;
    const int blk = local / (M_GROUP * NT);
    const int within = local - blk * M_GROUP * NT;
    const int bs = min(M_GROUP, cnt - blk * M_GROUP);
    nt = within / bs;
    mt = beg + blk * M_GROUP + (within - nt * bs);
  }
  int4 m = a.mt_info[mt];
  TileInfo t;
  t.slice = m.x;
  t.row0 = m.y;
  t.nrows = m.z;
  t.gbase = m.w;
  t.nt = nt;
  return t;
}

template <int MODE>
__device__ __forceinline__ int total_tiles(const TcGemmArgs& a) {
  if (MODE == kRouter) return ((a.n_rows + BM - 1) / BM) * a.n_ntiles;
  return a.group_mt_begin[a.n_groups] * a.n_ntiles;
}

// SiLU with the approximate divide (bf16 output: its 2-ulp error is far below the rounding;
// an IEEE divide per element made the SwiGLU epilogue outlast short main loops)
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ bool rows_identical(const __nv_bfloat16* rows, int d, int i, int j) {
  const uint4* a = reinterpret_cast<const uint4*>(rows + static_cast<long long>(i) * d);
  const uint4* b = reinterpret_cast<const uint4*>(rows + static_cast<long long>(j) * d);
  for (int v = 0; v < d / 8; ++v) {
    uint4 x = a[v], y = b[v];
    if (x.x != y.x || x.y != y.y || x.z != y.z || x.w != y.w) return false;
  }
  return true;
}

// Epilogue of one FFN tile for one TMEM lane (output row r of the tile): the
// SwiGLU tile writes h = SiLU(gate) * up, the store tile writes D, both bf16.
template <int MODE>
__device__ __forceinline__ void ffn_epilogue(const TcGemmArgs& args, const TileInfo& t,
                                             uint32_t col0, int r, bool valid) {
  if (MODE == kSwiGLU) {
    __nv_bfloat16* orow = args.out + (static_cast<long long>(t.row0) + r) * args.ld_out +
                          static_cast<long long>(t.nt) * (BN / 2);
#pragma unroll 1
    for (int c = 0; c < 4; ++c) {
      uint32_t g[32], u[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, g);
      ptx::tmem_ld_32x32b_x32(col0 + BN / 2 + c * 32, u);
      ptx::tmem_ld_wait();
      if (valid) {
        uint32_t p[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float h0 = silu_fast(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
          const float h1 =
              silu_fast(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
          p[i] = pack_bf16x2(h0, h1);
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
      }
    }
  } else {
    long long orow_idx = static_cast<long long>(t.row0) + r;
    if (valid && args.out_rowmap) orow_idx = args.out_rowmap[orow_idx];
    __nv_bfloat16* orow =
        args.out + orow_idx * args.ld_out + static_cast<long long>(t.nt) * BN;
#pragma unroll 1
    for (int c = 0; c < 8; c += 2) {
      uint32_t v0[32], v1[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, v0);
      ptx::tmem_ld_32x32b_x32(col0 + (c + 1) * 32, v1);
      ptx::tmem_ld_wait();
      if (valid) {
        uint32_t p[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          p[i] = pack_bf16x2(__uint_as_float(v0[2 * i]), __uint_as_float(v0[2 * i + 1]));
          p[16 + i] = pack_bf16x2(__uint_as_float(v1[2 * i]), __uint_as_float(v1[2 * i + 1]));
        }
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int v = 0; v < 8; ++v)
          dst[v] = make_uint4(p[4 * v], p[4 * v + 1], p[4 * v + 2], p[4 * v + 3]);
      }
    }
  }
}

// Epilogue of a full 32-row quarter of a pair tile (warp quarter q) through TMA: per
// 32-column chunk each thread writes its row's 64 bytes into a {32, 32} bf16 box in shared
// memory (64-byte swizzle: the row's four 16-byte pieces rotated by (row / 2) mod 4, so a
// quarter-warp's stores hit distinct banks) and one thread stores the box.  Two boxes per
// warp alternate; `nstore` counts the warp's stores.
template <int MODE>
__device__ __forceinline__ void ffn_epilogue_tma(const TcGemmArgs& args, const TileInfo& t,
                                                 uint32_t col0, int q, int lane, uint8_t* stage,
                                                 const CUtensorMap* tmO, uint32_t& nstore) {
  const int row = t.row0 + 32 * q;
  const int sw = (lane >> 1) & 3;
  constexpr int NCH = MODE == kSwiGLU ? 4 : 8;
  const int col_base = MODE == kSwiGLU ? t.nt * (BN / 2) : t.nt * BN;
#pragma unroll 1
  for (int c = 0; c < NCH; ++c) {
    uint32_t p[16];
    if (MODE == kSwiGLU) {
      uint32_t g[32], u[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, g);
      ptx::tmem_ld_32x32b_x32(col0 + BN / 2 + c * 32, u);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        p[i] = pack_bf16x2(silu_fast(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]),
                           silu_fast(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]));
    } else {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        p[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
    }
    if (lane == 0) ptx::bulk_wait_read1();  // the box written two stores ago has been read
    __syncwarp();
    uint8_t* box = stage + (nstore & 1u) * (32 * 32 * 2);
    uint8_t* mine = box + lane * 64;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      *reinterpret_cast<uint4*>(mine + ((j ^ sw) << 4)) =
          make_uint4(p[4 * j], p[4 * j + 1], p[4 * j + 2], p[4 * j + 3]);
    ptx::fence_proxy_async_smem_cta();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tmO, ptx::smem_u32(box), col_base + c * 32, row);
      ptx::bulk_commit();
    }
    ++nstore;
  }
}

// Tail tile of the CTA-pair kernel: the accumulator is transposed, TMEM lane =
// weight row of this CTA's 128-row half of the N tile, column = token of the
// tail (t.nrows <= kMaxTailRows of them).  Warp quarter q holds lanes [32q, 32q + 32).
//   kSwiGLU  lanes 32q + j (j < 16) are gate rows and lanes 32q + 16 + j the up
//            rows of hidden unit 64 rank + 16 q + j of the tile, so a lane and
//            its partner 16 apart swap half of each 32-token chunk: the low lane
//            ends with (gate, up) of tokens 0..15 of the chunk, the high lane
//            with those of tokens 16..31.
//   kStore   lane 32q + j is output column 128 rank + 32 q + j of the N tile.
template <int MODE>
__device__ __forceinline__ void tail_epilogue(const TcGemmArgs& args, const TileInfo& t,
                                              uint32_t col0, int q, int lane, uint32_t rank) {
  const int n = t.nrows;
  if (MODE == kSwiGLU) {
    const bool hi = lane >= 16;
    const long long col = static_cast<long long>(t.nt) * (BN / 2) + 64 * static_cast<int>(rank) +
                          16 * q + (lane & 15);
    __nv_bfloat16* out = args.out + col;
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += 32) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(col0 + c0, v);
      ptx::tmem_ld_wait();
      const int cb = c0 + (hi ? 16 : 0);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t other = __shfl_xor_sync(0xffffffffu, hi ? v[i] : v[16 + i], 16);
        const float g = __uint_as_float(hi ? other : v[i]);
        const float u = __uint_as_float(hi ? v[16 + i] : other);
        if (cb + i < n)
          out[(static_cast<long long>(t.row0) + cb + i) * args.ld_out] =
              __float2bfloat16_rn(silu_fast(g) * u);
      }
    }
  } else {
    const long long col = static_cast<long long>(t.nt) * BN + 128 * static_cast<int>(rank) +
                          32 * q + lane;
    __nv_bfloat16* out = args.out + col;
#pragma unroll 1
    for (int c0 = 0; c0 < n; c0 += 32) {
      uint32_t v[32];
      ptx::tmem_ld_32x32b_x32(col0 + c0, v);
      ptx::tmem_ld_wait();
      // lane i looks up the output row of token c0 + i
      long long my_row = static_cast<long long>(t.row0) + c0 + lane;
      if (args.out_rowmap && c0 + lane < n) my_row = args.out_rowmap[my_row];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const long long orow = __shfl_sync(0xffffffffu, my_row, i);
        if (c0 + i < n) out[orow * args.ld_out] = __float2bfloat16_rn(__uint_as_float(v[i]));
      }
    }
  }
}

// Operands of one Gram tile's epilogue that do not depend on the accumulator: the lane's
// row's inverse norm and hash (registers), and the 256 columns' {inverse norm, low hash
// word} (the warp's shared-memory slice, read by every lane as broadcasts).  Loaded before
// the wait on the accumulator, so their latency runs under the tile's MMAs.
struct SimOperands {
  float inv_ni;
  unsigned long long hi;
  float2* col;  // [256] shared: {1 / |x_j|, low word of x_j's hash as bits}
};

__device__ __forceinline__ void sim_prefetch(const TcGemmArgs& args, const TileInfo& t, int r,
                                             int lane, SimOperands& o) {
  const int e = t.slice;
  const int n_e = args.bucket_off[e + 1] - args.bucket_off[e];
  const bool valid = r < t.nrows;
  const float ni = valid ? args.norm[t.row0 + r] : 0.f;
  o.inv_ni = ni > 0.f ? 1.0f / ni : 0.f;
  o.hi = valid ? args.row_hash[t.row0 + r] : 0ull;
  float nj[BN / 32];
  uint32_t hj[BN / 32];
#pragma unroll
  for (int c = 0; c < BN / 32; ++c) {
    const int lj = t.nt * BN + c * 32 + lane;
    const bool col_in = lj < n_e;
    nj[c] = col_in ? args.norm[t.gbase + lj] : 0.f;
    hj[c] = col_in ? static_cast<uint32_t>(args.row_hash[t.gbase + lj]) : 0u;
  }
  __syncwarp();  // every lane is done with the previous tile's columns
#pragma unroll
  for (int c = 0; c < BN / 32; ++c)
    o.col[c * 32 + lane] = make_float2(nj[c] > 0.f ? 1.0f / nj[c] : 0.f, __uint_as_float(hj[c]));
  __syncwarp();
}

// Epilogue of one Gram tile of the similarity GEMM for one TMEM lane: row slot i = row0 + r
// of bucket e (valid: r < nrows), column slots j = gbase + nt * 256 + c, c < 256.  Writes
// the row's bit words of the tile and lowers first[i] to its earliest similar column.
__device__ __forceinline__ void sim_epilogue(const TcGemmArgs& args, const TileInfo& t,
                                             const SimOperands& o, uint32_t col0, int r,
                                             int lane) {
  // cos(x_i, x_j) = D[i][j] / (|x_i| |x_j|), taken as (D * (1/|x_i|)) * (1/|x_j|) in fp32,
  // clamped to [-1, 1]; a zero row has similarity 0 to every row it is not identical
  // to (its D and its inverse norm are 0), and identical rows have similarity exactly 1.
  // Bits: sim >= tau (the decision), and with history sim >= s1 / sim <= s2 (the classes
  // handed to the next call).  Without history only the decision is formed: the clamp is
  // then folded into it (tau <= 1 on this path, so min(s, 1) >= tau is s >= tau, and
  // max(s, -1) >= tau is s >= tau or tau <= -1).
  const int e = t.slice, gbase = t.gbase, nt = t.nt;
  const bool valid = r < t.nrows;
  const int n_e = args.bucket_off[e + 1] - args.bucket_off[e];
  const int W = (n_e + 31) >> 5;
  const int i = t.row0 + r;
  const int li = i - gbase;
  const float inv_ni = o.inv_ni;
  const unsigned long long hi = o.hi;
  const uint32_t hi_lo = static_cast<uint32_t>(hi);
  const long long wrow = args.bits_base[e] + static_cast<long long>(li) * W;
  unsigned* brow = args.bits + wrow;
  const int hmode = args.hist_mode;
  const float tau = args.tau;
  const bool all_similar = tau <= -1.f;
  const float4* col4 = reinterpret_cast<const float4*>(o.col);
  int hit = -1;  // earliest similar column of this tile (local index)
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int lj0 = nt * BN + c * 32;
    // a chunk that lies above every row of this warp's quarter holds no bit
    if (!__any_sync(0xffffffffu, valid && lj0 < li)) continue;
    uint32_t v[32];
    ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
    ptx::tmem_ld_wait();
    const int n_in = li - lj0;  // columns of this chunk below row li
    const uint32_t in_mask = n_in >= 32 ? 0xffffffffu : n_in <= 0 ? 0u : (1u << n_in) - 1u;
    uint32_t word = 0, w1 = 0, w2 = 0, same_hash = 0;
    if (hmode == 0) {
#pragma unroll
      for (int b = 0; b < 32; b += 2) {
        const float4 q = col4[c * 16 + (b >> 1)];  // columns b, b + 1 (a broadcast)
        const float s0 = __uint_as_float(v[b]) * inv_ni * q.x;
        const float s1 = __uint_as_float(v[b + 1]) * inv_ni * q.z;
        word |= (static_cast<uint32_t>(s0 >= tau) << b) | (static_cast<uint32_t>(s1 >= tau) << (b + 1));
        same_hash |= (static_cast<uint32_t>(__float_as_uint(q.y) == hi_lo) << b) |
                     (static_cast<uint32_t>(__float_as_uint(q.w) == hi_lo) << (b + 1));
      }
      if (all_similar) word = 0xffffffffu;
    } else {
#pragma unroll
      for (int b = 0; b < 32; b += 2) {
        const float4 q = col4[c * 16 + (b >> 1)];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float inv_nj = h ? q.z : q.x;
          const uint32_t hj_lo = __float_as_uint(h ? q.w : q.y);
          const float s = fminf(fmaxf(__uint_as_float(v[b + h]) * inv_ni * inv_nj, -1.f), 1.f);
          word |= static_cast<uint32_t>(s >= tau) << (b + h);
          w1 |= static_cast<uint32_t>(s >= args.s1) << (b + h);
          w2 |= static_cast<uint32_t>(s <= args.s2) << (b + h);
          same_hash |= static_cast<uint32_t>(hj_lo == hi_lo) << (b + h);
        }
      }
    }
    word &= in_mask;
    w1 &= in_mask;
    w2 &= in_mask;
    same_hash &= in_mask;
    // identical rows: similarity exactly 1 (full hash, then the rows themselves)
    while (valid && same_hash) {
      const int b = __ffs(same_hash) - 1;
      same_hash &= same_hash - 1;
      const int j = gbase + lj0 + b;
      if (args.row_hash[j] == hi && rows_identical(args.rows, args.d, i, j)) {
        const uint32_t m = 1u << b;
        word = 1.0f >= tau ? (word | m) : (word & ~m);
        w1 = 1.0f >= args.s1 ? (w1 | m) : (w1 & ~m);
        w2 = 1.0f <= args.s2 ? (w2 | m) : (w2 & ~m);
      }
    }
    if (valid && lj0 < li) {
      uint32_t wout = word;
      if (hmode != 0) {
        const long long widx = wrow + (lj0 >> 5);
        uint2 ks = make_uint2(0u, 0u);
        if (hmode == 2) ks = args.hplanes[widx];
        const uint32_t kw = ks.x, sw = ks.y;
        // a pair with a class is decided by it; the others by their cosine, and get
        // a class from it (similar first)
        wout = (kw & sw) | (~kw & word);
        args.hplanes[widx] = make_uint2(kw | (~kw & (w1 | w2)), (kw & sw) | (~kw & w1));
      }
      brow[lj0 >> 5] = wout;
      // the chunks run in column order: the first set bit is the tile's earliest similar row
      if (hit < 0 && wout) hit = lj0 + __ffs(wout) - 1;
    }
  }
  if (hit >= 0) atomicMin(&args.first[i], hit);
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB, const TcGemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  Shared* sh = reinterpret_cast<Shared*>(smem + STAGES * STAGE_BYTES);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem0 = ptx::smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(&sh->full[s]), 1);
      ptx::mbar_init(ptx::smem_u32(&sh->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_u32(&sh->tmem_full[a]), 1);
      ptx::mbar_init(ptx::smem_u32(&sh->tmem_empty[a]), 4);
    }
    ptx::mbar_init(ptx::smem_u32(&sh->drain), 1);
    sh->abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
  }
  // Barrier set-up above and TMEM allocation below touch no global memory, so
  // they overlap the previous kernel's tail; everything after waits for it.
  pdl_wait();
  if (MODE == kSwiGLU || MODE == kStore) {
    for (int g = threadIdx.x; g <= args.n_groups; g += blockDim.x)
      sh->gmb[g] = args.group_mt_begin[g];
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&sh->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = sh->tmem_base;
  const int n_tiles = total_tiles<MODE>(args);
  // Router with 65..128 experts: the three terms (up to 128 rows each) side by side need 64 KB
  // stages (three of them in the same ring), two MMAs per K step (terms 1 and 2, then term 3)
  // and a 384-column accumulator, so a single TMEM buffer.
  const bool wide = MODE == kRouter && args.router_stacked && 3 * args.router_n > BN;
  const int sbytes = wide ? WIDE_STAGE_BYTES : STAGE_BYTES;
  const int nst = wide ? WIDE_STAGES : STAGES;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    int stage = 0;
    uint32_t phase = 0;
    int issued[STAGES];
    uint32_t issued_phase[STAGES];
    for (int s = 0; s < STAGES; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
      const TileInfo t = tile_info<MODE>(args, sh->gmb, tile);
      for (int kb = 0; kb < args.n_kblocks; ++kb) {
        if (!wait_bar(ptx::smem_u32(&sh->empty[stage]), phase ^ 1u, sh, args.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = ptx::smem_u32(&sh->full[stage]);
          const uint32_t sa = smem0 + stage * sbytes;
          const uint32_t sb = sa + A_BYTES;
          const int kslice = kb / args.kb_per_slice;
          const int kin = (kb - kslice * args.kb_per_slice) * BK;
          if (MODE == kRouter && args.router_stacked) {
            // K block kb of this split: x once, the three terms' rows one after another
            const int k0 = (t.nt * args.n_kblocks + kb) * BK;
            ptx::mbar_arrive_expect_tx(full, A_BYTES + 3 * args.router_n * BK * 2);
            ptx::tma_load_2d(sa, &tmA, full, k0, t.row0);
#pragma unroll
            for (int term = 0; term < 3; ++term)
              ptx::tma_load_3d(sb + term * args.router_n * BK * 2, &tmB, full, k0, 0, term);
          } else if (MODE == kRouter) {
            // K block kb of this split -> term (W1, W2 or W3) and K offset inside x
            const int g = t.nt * args.n_kblocks + kb;
            const int term = g / args.router_kbd;
            const int k0 = (g - term * args.router_kbd) * BK;
            ptx::mbar_arrive_expect_tx(full, A_BYTES + args.router_n * BK * 2);
            ptx::tma_load_2d(sa, &tmA, full, k0, t.row0);
            ptx::tma_load_3d(sb, &tmB, full, k0, 0, term);
          } else {
            ptx::mbar_arrive_expect_tx(full, STAGE_BYTES);
            ptx::tma_load_2d(sa, &tmA, full, kb * BK, t.row0);
            if (MODE == kSwiGLU) {
              const int nslice = t.nt / args.nt_per_slice;
              const int n0 = (t.nt - nslice * args.nt_per_slice) * (BN / 2);
              const int z = t.slice + nslice + kslice;
              ptx::tma_load_3d(sb, &tmB, full, kin, n0, z);
              ptx::tma_load_3d(sb + B_BYTES / 2, &tmB, full, kin, args.b_up_offset + n0, z);
            } else if (MODE == kStore) {
              const int nslice = t.nt / args.nt_per_slice;
              const int n0 = (t.nt - nslice * args.nt_per_slice) * BN;
              ptx::tma_load_3d(sb, &tmB, full, kin, n0, t.slice + nslice + kslice);
            }
          }
        }
        __syncwarp();
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == nst) stage = 0, phase ^= 1u;
      }
    }
    if (!ok) {
      // Let the loads already in flight land before the CTA exits.
      for (int s = 0; s < nst; ++s) {
        if (!issued[s]) continue;
        uint64_t t0 = globaltimer_ns();
        while (!ptx::mbar_try_wait(ptx::smem_u32(&sh->full[s]), issued_phase[s]) &&
               globaltimer_ns() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t idesc = ptx::idesc_bf16_f32(
        BM, MODE == kRouter ? (wide ? 2 : args.router_stacked ? 3 : 1) * args.router_n : BN);
    const uint32_t idesc_term3 = ptx::idesc_bf16_f32(BM, MODE == kRouter ? args.router_n : BN);
    int stage = 0;
    uint32_t phase = 0;
    int local = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++local) {
      // one buffer when wide: its phase flips every tile
      const int acc = wide ? 0 : local & 1;
      const uint32_t acc_phase = wide ? local & 1 : (local >> 1) & 1;
      if (!wait_bar(ptx::smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1u, sh, args.status)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem_base + acc * BN;
      for (int kb = 0; kb < args.n_kblocks; ++kb) {
        if (!wait_bar(ptx::smem_u32(&sh->full[stage]), phase, sh, args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        if (lane == 0) {
          const uint32_t sa = smem0 + stage * sbytes;
          const uint32_t sb = sa + A_BYTES;
          const uint64_t adesc = ptx::sw128_kmajor_desc(sa);
          const uint64_t bdesc = ptx::sw128_kmajor_desc(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            // +32 bytes per K step of 16 elements = +2 in the encoded start address
            ptx::umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                           (kb > 0 || kk > 0) ? 1u : 0u);
          }
          if (wide) {
            // the third term's rows, into the columns after the first two terms'
            const uint64_t bdesc3 = ptx::sw128_kmajor_desc(sb + 2 * args.router_n * BK * 2);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              ptx::umma_bf16(d_tmem + 2 * args.router_n, adesc + 2 * kk, bdesc3 + 2 * kk,
                             idesc_term3, (kb > 0 || kk > 0) ? 1u : 0u);
          }
          ptx::umma_commit(ptx::smem_u32(&sh->empty[stage]));
        }
        __syncwarp();
        if (++stage == nst) stage = 0, phase ^= 1u;
      }
      if (!ok) break;
      if (lane == 0) ptx::umma_commit(ptx::smem_u32(&sh->tmem_full[acc]));
      __syncwarp();
    }
    if (!ok) {
      // Wait for the MMAs already issued before TMEM is released.
      if (lane == 0) ptx::umma_commit(ptx::smem_u32(&sh->drain));
      __syncwarp();
      uint64_t t0 = globaltimer_ns();
      while (!ptx::mbar_try_wait(ptx::smem_u32(&sh->drain), 0) &&
             globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int local = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++local) {
      const int acc = wide ? 0 : local & 1;
      const uint32_t acc_phase = wide ? local & 1 : (local >> 1) & 1;
      if (!wait_bar(ptx::smem_u32(&sh->tmem_full[acc]), acc_phase, sh, args.status)) break;
      ptx::tc_fence_after();
      const TileInfo t = tile_info<MODE>(args, sh->gmb, tile);
      const uint32_t col0 = lane_addr + acc * BN;
      const bool valid = r < t.nrows;
      if (MODE == kRouter) {
        float* prow = args.part + (static_cast<long long>(t.nt) * args.n_rows + t.row0 + r) *
                                      args.router_n;
#pragma unroll 1
        for (int c = 0; c < args.router_n / 32; ++c) {
          uint32_t v[32];
          ptx::tmem_ld_32x32b_x32(col0 + c * 32, v);
          if (args.router_stacked) {
            // the three terms' accumulators, the two small ones added first
            uint32_t v1[32], v2[32];
            ptx::tmem_ld_32x32b_x32(col0 + args.router_n + c * 32, v1);
            ptx::tmem_ld_32x32b_x32(col0 + 2 * args.router_n + c * 32, v2);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[i] = __float_as_uint(__uint_as_float(v[i]) +
                                     (__uint_as_float(v1[i]) + __uint_as_float(v2[i])));
          }
          ptx::tmem_ld_wait();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(prow + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                   __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
          }
        }
      } else if (MODE == kSwiGLU || MODE == kStore) {
        ffn_epilogue<MODE>(args, t, col0, r, valid);
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sh->tmem_empty[acc]));
    }
  }

  // This CTA's work is done: the next kernel on the stream may be scheduled.
  pdl_trigger();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- CTA-pair kernel
// The FFN GEMMs on pairs of SMs (clusters of two CTAs, tcgen05 cta_group::2).
// A pair tile is 256 rows x 256 columns: CTA r of the pair holds rows
// [128 r, 128 r + 128) of A and the r-th 128-row half of the B tile (gate rows
// then up rows for the SwiGLU tile), so a 64-deep K block is 32 KB per SM instead
// of 48 KB.  A ring stage holds two K blocks (three stages of 64 KB): the MMA
// issuer's barrier wait and commit, which cost the tensor pipe far more than an
// MMA's issue, come once per 8 MMAs.  The even (leader) CTA issues M=256 x N=256
// MMAs that read both CTAs' shared memory and write each CTA's own TMEM rows; each
// CTA runs its own epilogue exactly as the single-CTA kernel does.
//   full[s]       leader only; both CTAs' TMA loads complete on it (128 KB)
//   empty[s]      both CTAs; the leader's MMA commit arrives on both
//   tmem_full[a]  both CTAs; the leader's commit arrives on both
//   tmem_empty[a] leader only; 4 epilogue warps of each CTA arrive (8)
// A pair tile is two consecutive m-tiles of one group.  When a group's rows after its
// full pairs are at most kMaxTailRows (192), they run as a tail tile with the roles of
// the operands swapped: A is the 256 weight rows of the N tile (128 per CTA), B is the
// left-over rows (N = their count rounded up to 16, half in each CTA, one 64- or
// 128-row box), so D is transposed in TMEM.  The tail's MMAs cost in proportion to
// its rows, where a partial pair's cost a full 256; and it loads no token rows past
// the group's end.  More rows left than that run as one more (partial) pair.
//   kSwiGLU tail A rows, per CTA: for q = 0..3, 16 gate rows then 16 up rows
//           of hidden units 64 rank + 16 q + [0, 16) of the tile (tail_epilogue),
//           one TMA box of a 5-D view of the gate/up weights.
//   kStore  tail A rows: the same 128 weight rows the CTA loads as B in a pair tile.
namespace pr {
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = (BN / 2) * BK * 2;
// A ring stage holds KSUB consecutive 64-deep K blocks (each laid out as A then B, as one
// 32 KB block): the MMA issuer waits once and commits once per stage, for 4 x KSUB MMAs.
constexpr int KSUB = 2;
constexpr int SUB_BYTES = A_BYTES + B_BYTES;
constexpr int STAGE_BYTES = KSUB * SUB_BYTES;
constexpr int STAGES = 6 / KSUB;
constexpr int SHARED_BYTES = 5120;
// per epilogue warp: two {32 columns, 32 rows} bf16 TMA store boxes of 2 KB (64-byte swizzle)
constexpr int OUT_BOX_BYTES = 32 * 32 * 2;
constexpr int OUT_STAGE_BYTES = 4 * 2 * OUT_BOX_BYTES;
static_assert(2 * BN * 4 <= 2 * OUT_BOX_BYTES, "a warp's similarity operands fit its staging area");
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + SHARED_BYTES + OUT_STAGE_BYTES;
static_assert((STAGES * STAGE_BYTES + SHARED_BYTES) % 1024 == 0, "output boxes 1024-byte aligned");
// Units per block of the tile walk.  Measured on the Llama-4-Scout-shaped shared expert
// (32 pair tiles, K = 5120): blocks of 8 keep the block's 21 MB of token rows in L2 and read
// the weights once per block; blocks of 25 (65 MB of token rows) lost the rows from L2 and
// read 1.84x the DRAM bytes.
constexpr int kUnitGroup = 8;
constexpr int TAIL_ROWS = BM / 2;  // token rows a CTA loads for a tail tile (box height)
// Rows left after a group's full pairs that run as a tail tile (weights as M, the rows as N,
// so its MMAs cost in proportion to the rows) rather than as a partial pair: up to 192;
// a tail of more than 128 rows loads its half of them with the 128-row box.
constexpr int kMaxTailRows = 192;
constexpr int TAIL_W_ROWS = 16;    // hidden units per gate (or up) run of a kSwiGLU tail
constexpr int TAIL_TX = 2 * (A_BYTES + TAIL_ROWS * BK * 2);  // both CTAs, one K block
constexpr int TAIL_TX_BIG = 2 * (A_BYTES + BM * BK * 2);      // the same with the 128-row box
// Launches whose every group is a tail of at most 128 rows (batches of at most 128 tokens):
// a K block needs only the weights and a 64-row token box, 24 KB, so four stages of two K
// blocks fit where three of the general layout do.
constexpr int TAIL_SUB_BYTES = A_BYTES + TAIL_ROWS * BK * 2;
constexpr int STAGES_TAILS = 4;
static_assert(STAGES_TAILS * KSUB * TAIL_SUB_BYTES == STAGES * STAGE_BYTES, "one layout size");
static_assert(TAIL_SUB_BYTES % 1024 == 0, "1024-byte aligned K blocks");
template <bool TAILS> __host__ __device__ constexpr int sub_bytes() { return TAILS ? TAIL_SUB_BYTES : SUB_BYTES; }
template <bool TAILS> __host__ __device__ constexpr int n_stages() { return TAILS ? STAGES_TAILS : STAGES; }
static_assert(TAIL_ROWS * BK * 2 <= B_BYTES, "tail tokens fit the B region");
static_assert(TAIL_ROWS == kTailOnlyRows, "tails-only launches hold tails of 2 x TAIL_ROWS rows");
static_assert(kMaxTailRows <= 2 * BM && BM * BK * 2 <= B_BYTES, "a big tail's half fits the B region");
// Token rows each CTA of the pair provides for a tail tile of n rows (N = n rounded up to 16).
__host__ __device__ constexpr int tail_half(int n) { return ((n + 15) & ~15) >> 1; }
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");

constexpr int MAX_STAGES = STAGES_TAILS > STAGES ? STAGES_TAILS : STAGES;

struct Shared {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int abort_flag;
  int goff[257];   // first row of each group
  int grows[256];  // rows of each group
  int gub[257];    // first unit (pair or tail) of each group
  int gpt[256];    // pairs of each group | rows of its tail (0..kMaxTailRows) << 16
};
static_assert(sizeof(Shared) <= SHARED_BYTES, "pair kernel barriers and tables");

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

// Tile -> this CTA's part.  Groups are walked in order; inside a group, blocks
// of a.unit_group units (pairs first, then tails), N tiles with the units
// fastest, so a group's tails run beside its pairs and share their weights in L2,
// and a block's token rows stay in L2 while the weights stream past them.  Odd blocks walk
// the N tiles in reverse, so a block starts on the weight tiles the block before it used
// last, which are still in L2 (a group's weights can be larger than L2: the shared expert's
// gate/up projection of the Llama-4-Scout-shaped layer is 168 MB).
__device__ __forceinline__ TileInfo tile_info(const TcGemmArgs& a, const Shared* sh, int tile,
                                              uint32_t rank) {
  const int NT = a.n_ntiles;
  int lo = 0, hi = a.n_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (sh->gub[mid] * NT <= tile) lo = mid; else hi = mid;
  }
  const int beg = sh->gub[lo], cnt = sh->gub[lo + 1] - beg;
  const int local = tile - beg * NT;
  const int G = a.unit_group;
  const int blk = local / (G * NT);
  const int within = local - blk * G * NT;
  const int bs = min(G, cnt - blk * G);
  const int nt_fwd = within / bs;
  const int u = blk * G + (within - nt_fwd * bs);
  const int nt = (blk & 1) ? NT - 1 - nt_fwd : nt_fwd;
  const int np = sh->gpt[lo] & 0xffff;
  const bool tail = u >= np;
  // m-tile of the group: 128-row tile 2u + rank of a pair, or the one left after the pairs
  const int mt = tail ? 2 * np : 2 * u + static_cast<int>(rank);
  TileInfo t;
  t.nt = nt;
  t.slice = lo;
  t.gbase = sh->goff[lo];
  t.row0 = t.gbase + mt * BM;
  t.nrows = tail ? sh->gpt[lo] >> 16 : min(BM, sh->grows[lo] - mt * BM);
  t.tail = tail ? 1 : 0;
  return t;
}

// Similarity tile -> this CTA's part: tile_list[tile] = {first m-tile of a pair of a bucket's
// m-tiles, column tile | (1 << 16) when the pair's second m-tile is in the same bucket}.  CTA
// rank r takes m-tile r of the pair (no rows when the bucket has only the first).
__device__ __forceinline__ TileInfo sim_tile_info(const TcGemmArgs& a, int tile, uint32_t rank) {
  const int2 e = a.tile_list[tile];
  const int4 m0 = a.mt_info[e.x];
  TileInfo t;
  t.slice = m0.x;
  t.gbase = m0.w;
  t.nt = e.y & 0xffff;
  t.tail = 0;
  if (rank == 0) {
    t.row0 = m0.y;
    t.nrows = m0.z;
  } else if ((e.y >> 16) & 1) {
    const int4 m1 = a.mt_info[e.x + 1];
    t.row0 = m1.y;
    t.nrows = m1.z;
  } else {
    t.row0 = m0.y + BM;
    t.nrows = 0;
  }
  return t;
}

// This CTA's loads of K block kb, completing on the leader's barrier `full`:
// for a pair tile its A rows and its half of the B tile; for a tail tile its
// 128 weight rows (into the A region) and its half of the tail's token rows
// (into the B region).
template <int MODE>
__device__ __forceinline__ void issue_kblock(const TcGemmArgs& args, const CUtensorMap* tmA,
                                             const CUtensorMap* tmB, const CUtensorMap* tmA64,
                                             const CUtensorMap* tmW5, const TileInfo& t, int kb,
                                             uint32_t rank, uint32_t full, uint32_t sa,
                                             uint32_t sb) {
  if (MODE == kSimBits) {
    // the bucket's rows: A = this CTA's 128 rows i, B = its half of the 256 column rows j
    ptx::tma_load_2d_pair(sa, tmA, full, kb * BK, t.row0);
    ptx::tma_load_3d_pair(sb, tmB, full, kb * BK,
                          t.gbase + t.nt * BN + static_cast<int>(rank) * (BN / 2), 0);
    return;
  }
  const int kslice = kb / args.kb_per_slice;
  const int kin = (kb - kslice * args.kb_per_slice) * BK;
  const int nslice = t.nt / args.nt_per_slice;
  const int z = t.slice + nslice + kslice;
  if (t.tail) {
    const int half = tail_half(t.nrows);
    ptx::tma_load_2d_pair(sb, half <= TAIL_ROWS ? tmA64 : tmA, full, kb * BK,
                          t.row0 + static_cast<int>(rank) * half);
  } else {
    ptx::tma_load_2d_pair(sa, tmA, full, kb * BK, t.row0);
  }
  const uint32_t dw = t.tail ? sa : sb;  // the weights' region
  if (MODE == kSwiGLU) {
    const int ntl = (t.nt - nslice * args.nt_per_slice) * (BN / 2);
    if (t.tail) {
      // box {64 K, 16 units, gate|up, 4 runs}: smem rows [q][gate|up][16]
      ptx::tma_load_5d_pair(dw, tmW5, full, kin, 0, 0,
                            (ntl + 64 * static_cast<int>(rank)) / TAIL_W_ROWS, z);
    } else {
      ptx::tma_load_3d_pair(dw, tmB, full, kin, (rank ? args.b_up_offset : 0) + ntl, z);
    }
  } else {
    const int n0 = (t.nt - nslice * args.nt_per_slice) * BN + static_cast<int>(rank) * (BN / 2);
    ptx::tma_load_3d_pair(dw, tmB, full, kin, n0, z);
  }
}
}  // namespace pr

template <int MODE, bool TAILS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                             const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmA64,
                             const __grid_constant__ CUtensorMap tmW5,
                             const __grid_constant__ CUtensorMap tmO, const TcGemmArgs args) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  constexpr int NS = pr::n_stages<TAILS>();
  constexpr int SUBB = pr::sub_bytes<TAILS>();
  constexpr int SB = pr::KSUB * SUBB;
  pr::Shared* sh = reinterpret_cast<pr::Shared*>(smem + NS * SB);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const uint32_t smem0 = ptx::smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
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
    ptx::prefetch_tmap(&tmA64);
    ptx::prefetch_tmap(&tmW5);
    ptx::prefetch_tmap(&tmO);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&sh->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();  // both CTAs' barriers and the pair's TMEM exist from here on
  ptx::tc_fence_after();
  pdl_wait();
  // Rows of each group, from the group offsets, from a fixed row count, or from the m-tile
  // table (whose m-tiles are 128-row pieces of each group from its first row).  Units of each
  // group: pairs of m-tiles, then a tail if a single m-tile is left.  (The similarity tiles
  // come from an explicit list instead.)
  for (int g = threadIdx.x; MODE != kSimBits && g < args.n_groups; g += blockDim.x) {
    int off = 0, rows = 0;
    if (args.group_off) {
      off = args.group_off[g];
      rows = args.group_off[g + 1] - off;
    } else if (args.fixed_rows > 0) {
      off = g * args.fixed_rows;
      rows = args.fixed_rows;
    } else {
      const int b = args.group_mt_begin[g], e = args.group_mt_begin[g + 1];
      if (e > b) {
        const int4 first = args.mt_info[b];
        off = first.w;
        rows = (e - b - 1) * BM + args.mt_info[e - 1].z;
      }
    }
    // full pairs, then the rows left: up to kMaxTailRows run as a tail tile (its MMA's N is
    // their count), more as one more (partial) pair
    const int full = rows / (2 * BM);
    const int left = rows - full * 2 * BM;
    const bool as_tail = left > 0 && left <= pr::kMaxTailRows;
    const int np = full + (left > 0 && !as_tail ? 1 : 0);
    const int tail_rows = as_tail ? left : 0;
    sh->goff[g] = off;
    sh->grows[g] = rows;
    // a tails-only launch takes no pair and no tail of more than 128 rows (the host picks it
    // for batches of at most 128 tokens; any other offsets are refused below)
    if (TAILS && (np > 0 || tail_rows > 2 * pr::TAIL_ROWS)) sh->abort_flag = 1;
    sh->gpt[g] = np | (tail_rows << 16);
    sh->gub[g] = np + (tail_rows > 0 ? 1 : 0);  // units, turned into offsets below
  }
  __syncthreads();
  if (MODE != kSimBits && warp == 0) {
    // exclusive scan of the unit counts, lane l owning groups [8 l, 8 l + 8)
    const int per = (args.n_groups + 31) >> 5;
    const int g0 = lane * per;
    int sum = 0;
    for (int i = 0; i < per; ++i)
      if (g0 + i < args.n_groups) sum += sh->gub[g0 + i];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - sum;
    __syncwarp();
    for (int i = 0; i < per; ++i) {
      if (g0 + i < args.n_groups) {
        const int c = sh->gub[g0 + i];
        sh->gub[g0 + i] = run;
        run += c;
      }
    }
    if (lane == 31) sh->gub[args.n_groups] = incl;
  }
  __syncthreads();
  const uint32_t tmem_base = sh->tmem_base;
  int n_tiles = MODE == kSimBits ? *args.n_list : sh->gub[args.n_groups] * args.n_ntiles;
  if (TAILS && sh->abort_flag) {
    // offsets this layout cannot take: no tile runs, the status word says why
    if (threadIdx.x == 0) record_status(args.status, MOE_ERR_DEVICE_INDEX);
    n_tiles = 0;
  }
  const int cluster = blockIdx.x >> 1, n_clusters = gridDim.x >> 1;
  auto tile_of = [&](int tile, uint32_t r) {
    return MODE == kSimBits ? pr::sim_tile_info(args, tile, r) : pr::tile_info(args, sh, tile, r);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int tile = cluster; tile < n_tiles && ok; tile += n_clusters) {
      const TileInfo t = tile_of(tile, rank);
      for (int kb0 = 0; kb0 < args.n_kblocks; kb0 += pr::KSUB) {
        const int nsub = min(pr::KSUB, args.n_kblocks - kb0);
        if (!pr::wait_bar(ptx::smem_u32(&sh->empty[stage]), phase ^ 1u, sh, args.status)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          const uint32_t full = ptx::smem_u32(&sh->full[stage]) & ptx::kLeaderMask;
          const uint32_t sbase = smem0 + stage * SB;
          if (rank == 0)
            ptx::mbar_arrive_expect_tx(
                full, nsub * (!t.tail                           ? 2 * pr::SUB_BYTES
                              : pr::tail_half(t.nrows) <= pr::TAIL_ROWS ? pr::TAIL_TX
                                                                        : pr::TAIL_TX_BIG));
          if (!fault_drop_loads())
            for (int u = 0; u < nsub; ++u) {
              const uint32_t sa = sbase + u * SUBB;
              pr::issue_kblock<MODE>(args, &tmA, &tmB, &tmA64, &tmW5, t, kb0 + u, rank, full, sa,
                                     sa + pr::A_BYTES);
            }
        }
        __syncwarp();
        if (++stage == NS) stage = 0, phase ^= 1u;
      }
    }
    if (!ok) {
      // give loads already issued time to land (microseconds) before the pair exits
      const uint64_t t0 = globaltimer_ns();
      while (globaltimer_ns() - t0 < 200000ull) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (rank == 0) {
      const uint32_t idesc_pair = ptx::idesc_bf16_f32(2 * BM, BN);
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      // the next ring stage's full barrier, tested before this stage's MMAs are issued: a
      // blocking wait on a barrier that has already completed holds the issuer about 200
      // cycles, during which the tensor pipe runs dry
      uint32_t next_ready = 0;
      for (int tile = cluster; tile < n_tiles && ok; tile += n_clusters, ++local) {
        const TileInfo t = tile_of(tile, 0);
        const uint32_t idesc =
            t.tail ? ptx::idesc_bf16_f32(2 * BM, (t.nrows + 15) & ~15) : idesc_pair;
        const int acc = local & 1;
        const uint32_t acc_phase = (local >> 1) & 1;
        if (!pr::wait_bar(ptx::smem_u32(&sh->tmem_empty[acc]), acc_phase ^ 1u, sh, args.status)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb0 = 0; kb0 < args.n_kblocks; kb0 += pr::KSUB) {
          const int nsub = min(pr::KSUB, args.n_kblocks - kb0);
          if (!next_ready &&
              !pr::wait_bar(ptx::smem_u32(&sh->full[stage]), phase, sh, args.status)) {
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          {
            const int ns = stage + 1 == NS ? 0 : stage + 1;
            next_ready = ptx::mbar_test_wait(ptx::smem_u32(&sh->full[ns]), ns ? phase : phase ^ 1u);
          }
          if (lane == 0) {
            for (int u = 0; u < nsub; ++u) {
              const uint32_t sa = smem0 + stage * SB + u * SUBB;
              const uint64_t adesc = ptx::sw128_kmajor_desc(sa);
              const uint64_t bdesc = ptx::sw128_kmajor_desc(sa + pr::A_BYTES);
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk)
                ptx::umma_bf16_pair(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, idesc,
                                    (kb0 + u > 0 || kk > 0) ? 1u : 0u);
            }
            ptx::umma_commit_pair(ptx::smem_u32(&sh->empty[stage]), 0x3);
          }
          __syncwarp();
          if (++stage == NS) stage = 0, phase ^= 1u;
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
    // full quarters store through TMA boxes, except a down projection with remapped rows
    uint8_t* out_stage = smem + NS * SB + pr::SHARED_BYTES +
                         (warp - 2) * 2 * pr::OUT_BOX_BYTES;
    const bool tma_out = MODE == kSwiGLU || args.out_rowmap == nullptr;
    uint32_t nstore = 0;
    int local = 0;
    for (int tile = cluster; tile < n_tiles; tile += n_clusters, ++local) {
      const int acc = local & 1;
      const uint32_t acc_phase = (local >> 1) & 1;
      const TileInfo t = tile_of(tile, rank);
      SimOperands so;
      if (MODE == kSimBits) {
        // the warp's output staging area is free in this mode
        so.col = reinterpret_cast<float2*>(out_stage);
        sim_prefetch(args, t, r, lane, so);
      }
      if (!pr::wait_bar(ptx::smem_u32(&sh->tmem_full[acc]), acc_phase, sh, args.status)) break;
      ptx::tc_fence_after();
      if (MODE == kSimBits) sim_epilogue(args, t, so, lane_addr + acc * BN, r, lane);
      else if (t.tail) tail_epilogue<MODE>(args, t, lane_addr + acc * BN, q, lane, rank);
      else if (tma_out && 32 * q + 32 <= t.nrows)
        ffn_epilogue_tma<MODE>(args, t, lane_addr + acc * BN, q, lane, out_stage, &tmO, nstore);
      else ffn_epilogue<MODE>(args, t, lane_addr + acc * BN, r, r < t.nrows);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t e = ptx::smem_u32(&sh->tmem_empty[acc]);
        if (rank == 0) ptx::mbar_arrive(e);
        else ptx::mbar_arrive_cluster(ptx::mapa(e, 0));
      }
    }
    if (lane == 0) ptx::bulk_wait0();  // this warp's output stores are performed
    __syncwarp();
  }

  pdl_trigger();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();  // the leader's MMAs into this CTA's TMEM and all remote arrivals are done
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 tensor map with 128-byte swizzle and a box of 64 (K) x box_rows.
// rank 2: [rows][inner]; rank 3: [outer][rows][inner].
static bool make_map(CUtensorMap* m, int rank, const void* base, uint64_t inner, uint64_t rows,
                     uint64_t outer, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {inner, rows, outer};
  cuuint64_t strides[2] = {inner * 2, inner * rows * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(BK), box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                  strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 5-D view of gate/up weights [slices][2H][K] for the kSwiGLU tail tiles:
// {K, unit in a run of 16, gate|up, run, slice}, box {64, 16, 2, 4, 1}, so one
// load puts, for four runs of 16 hidden units, 16 gate rows then 16 up rows.
static bool make_gate_up_map(CUtensorMap* m, const void* base, uint64_t K, uint64_t H,
                             uint64_t slices) {
  auto fn = encode_fn();
  if (!fn || H % pr::TAIL_W_ROWS != 0) return false;
  const uint64_t row = K * 2;
  cuuint64_t dims[5] = {K, static_cast<cuuint64_t>(pr::TAIL_W_ROWS), 2, H / pr::TAIL_W_ROWS,
                        slices};
  cuuint64_t strides[4] = {row, H * row, pr::TAIL_W_ROWS * row, 2 * H * row};
  cuuint32_t box[5] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(pr::TAIL_W_ROWS), 2,
                       4, 1};
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides,
                  box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 output [rows][inner] for TMA stores of {32, 32} boxes, 64-byte swizzle
static bool make_out_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t es[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, bool TAILS>
static cudaError_t launch_pair(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& a64,
                               const CUtensorMap& w5, const CUtensorMap& o, const TcGemmArgs& args,
                               int num_sms,
                               cudaStream_t stream) {
  static OncePerDevice<64> once;
  static int max_clusters[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  cudaLaunchConfig_t cfg = {};
  const cudaError_t set_up = once.run(dev, [&]() -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE, TAILS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         pr::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // Pairs of SMs that can hold a cluster at once: the persistent grid uses no more.
    cudaLaunchAttribute ca;
    ca.id = cudaLaunchAttributeClusterDimension;
    ca.val.clusterDim.x = 2;
    ca.val.clusterDim.y = 1;
    ca.val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * (num_sms / 2));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = pr::SMEM_BYTES;
    cfg.attrs = &ca;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<MODE, TAILS>, &cfg) !=
            cudaSuccess ||
        n <= 0)
      n = num_sms / 2;
    if (dev < 64) max_clusters[dev] = n;
    return cudaSuccess;
  });
  if (set_up != cudaSuccess) return set_up;
  const int clusters = dev < 64 ? (max_clusters[dev] < num_sms / 2 ? max_clusters[dev] : num_sms / 2)
                                : num_sms / 2;
  cfg = cudaLaunchConfig_t{};
  cfg.gridDim = dim3(2 * clusters);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = pr::SMEM_BYTES;
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
  return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE, TAILS>, a, b, a64, w5, o, args);
}

template <int MODE>
static cudaError_t launch(const CUtensorMap& a, const CUtensorMap& b, const TcGemmArgs& args,
                          int grid, cudaStream_t stream) {
  static OncePerDevice<64> once;
  int dev = 0;
  cudaGetDevice(&dev);
  const cudaError_t e = once.run(dev, [&]() {
    return cudaFuncSetAttribute(grouped_gemm_kernel<MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(grouped_gemm_kernel<MODE>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream, a,
                    b, args);
}

}  // namespace tc

#ifdef MOE_FAULT_INJECTION
// Test build only: switch the dropped loads on (1) or off (0) on the current device.
extern "C" int moe_test_drop_gemm_loads(int on) {
  const int v = on ? 1 : 0;
  return cudaMemcpyToSymbol(tc::g_fault_drop_loads, &v, sizeof(v)) == cudaSuccess ? 0 : 4;
}
#endif

cudaError_t tc_gemm(int mode, const void* A, long long a_rows, int K, const void* B,
                    int b_slices, int b_rows, int b_cols, const TcGemmArgs& args_in, int grid,
                    cudaStream_t stream) {
  CUtensorMap ma, mb;
  TcGemmArgs args = args_in;
  if (args.unit_group <= 0) args.unit_group = tc::pr::kUnitGroup;
  if (!tc::make_map(&ma, 2, A, K, a_rows, 1, tc::BM)) return cudaErrorInvalidValue;
  // The FFN and similarity modes run on CTA pairs, each CTA loading half of the 256-row B tile.
  const bool ffn = mode == tc::kSwiGLU || mode == tc::kStore;
  const bool pair = ffn || mode == tc::kSimBits;
  const uint32_t box_rows = pair                  ? tc::BN / 2
                            : mode == tc::kRouter ? static_cast<uint32_t>(args.router_n)
                                                  : tc::BN;
  if (!tc::make_map(&mb, 3, B, b_cols, b_rows, b_slices, box_rows)) return cudaErrorInvalidValue;
  // Tail tiles: a 64-row token box, and for kSwiGLU the interleaved gate/up view.
  CUtensorMap ma64, mw5 = mb;
  if (pair && !tc::make_map(&ma64, 2, A, K, a_rows, 1, tc::pr::TAIL_ROWS))
    return cudaErrorInvalidValue;
  if (mode == tc::kSwiGLU && !tc::make_gate_up_map(&mw5, B, b_cols, args.b_up_offset, b_slices))
    return cudaErrorInvalidValue;
  // the output [a_rows][ld_out] bf16, stored in {32, 32} boxes by the full-quarter epilogue
  CUtensorMap mo = ma;
  if (ffn && !tc::make_out_map(&mo, args.out, static_cast<uint64_t>(args.ld_out),
                               static_cast<uint64_t>(a_rows)))
    return cudaErrorInvalidValue;
  switch (mode) {
    case tc::kSwiGLU:
      return args.tails_only
                 ? tc::launch_pair<tc::kSwiGLU, true>(ma, mb, ma64, mw5, mo, args, grid, stream)
                 : tc::launch_pair<tc::kSwiGLU, false>(ma, mb, ma64, mw5, mo, args, grid, stream);
    case tc::kStore:
      return args.tails_only
                 ? tc::launch_pair<tc::kStore, true>(ma, mb, ma64, mw5, mo, args, grid, stream)
                 : tc::launch_pair<tc::kStore, false>(ma, mb, ma64, mw5, mo, args, grid, stream);
    case tc::kSimBits:
      return tc::launch_pair<tc::kSimBits, false>(ma, mb, ma64, mw5, mo, args, grid, stream);
    case tc::kRouter: return tc::launch<tc::kRouter>(ma, mb, args, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
