// Internal (C++) launch interface between the C-ABI layer (moe_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ------------------------------------------------------------------ router
// fp32 layers: logits = x W_r (+bias) in fp32 FMA.
cudaError_t launch_router_logits(int act_dtype, const void* x, const float* W_r, const float* bias,
                                 float* logits, int T, int d, int E, cudaStream_t stream);
// bf16 layers: W_r [d,E] fp32 -> W3 [3][E_pad][d] bf16 with W_r = W1 + W2 + W3 exactly,
// then the tcgen05 GEMM writes split-K partial logits.
int router_n_pad(int E);
int router_splits(int T, int d, int E, int num_sms);
size_t router_scratch_bytes(int T, int d, int E, int num_sms);
cudaError_t launch_router_tc(const void* x, const float* W_r, int T, int d, int E, int num_sms,
                             void* scratch, const float** part, int* n_split, int* ld,
                             unsigned* status, cudaStream_t stream);
// logits[t,e] = sum_s part[s][t][e] (s in order) + bias[e]; then top-k and gates.
// logits_out may be NULL (or equal to part when n_split == 1 and bias == NULL).
cudaError_t launch_router_topk(const float* part, int n_split, int ld, const float* bias,
                               float* logits_out, int32_t* topk_idx, float* topk_gate, int T,
                               int E, int k, int gating, cudaStream_t stream);

// ------------------------------------------------------------------ dispatch / combine
constexpr int kDispatchChunk = 128;  // tokens per dispatch chunk
size_t dispatch_scratch_bytes(int T, int E);
cudaError_t launch_dispatch(int act_dtype, const void* x, const int32_t* topk_idx, int T, int d,
                            int E, int k, int32_t* counts, int32_t* offsets, int32_t* perm,
                            int32_t* slot_of, void* x_perm, void* scratch, unsigned* status,
                            cudaStream_t stream);
// Same outputs as launch_dispatch, with ranks computed in parallel blocks of
// 1024 pairs; scratch: dispatch_auto_scratch_bytes.
size_t dispatch_auto_scratch_bytes(int T, int k, int E);
// Condensation row statistics at the slots (bf16 only): norm and hash as the condensation's
// row-statistics pass forms them, and the earliest-similar-row entry reset to kNoHit.
struct RowStatsOut {
  float* norm;
  unsigned long long* hash;
  int32_t* first;
};
constexpr int32_t kNoHit = 0x7fffffff;
// stats (nullable): the dispatch also writes each slot's row statistics (condense_stats_ptrs
// gives where the condensation reads them).
cudaError_t launch_dispatch_auto(int act_dtype, const void* x, const int32_t* topk_idx, int T,
                                 int d, int E, int k, int32_t* counts, int32_t* offsets,
                                 int32_t* perm, int32_t* slot_of, void* x_perm, void* scratch,
                                 int num_sms, unsigned* status, cudaStream_t stream,
                                 const RowStatsOut* stats = nullptr);
// dst[r] = src[rows[r]] for r < *n_rows_dev (<= max_rows); rows outside [0, src_rows) are flagged.
cudaError_t launch_gather_rows(int act_dtype, const void* src, int src_rows, const int32_t* rows,
                               const int* n_rows_dev, int max_rows, int d, void* dst,
                               unsigned* status, cudaStream_t stream);
// partial (nullable): also writes p = r + shared_out, the sum before the routed terms.
// inputs_ready: x and residual were complete before the previous kernel on the stream
// started (true only inside the layer's own launch chain); they are then read before the
// programmatic-launch wait.
cudaError_t launch_combine(int act_dtype, const void* y_perm, const void* shared_out,
                           const int32_t* slot_of, const int32_t* rep_of, const float* topk_gate,
                           const void* x, const void* residual, int residual_mode, void* out, int T,
                           int d, int k, int P, unsigned* status, cudaStream_t stream,
                           void* partial = nullptr, bool inputs_ready = false);

// ------------------------------------------------------------------ m-tile tables
// Groups of rows (experts, buckets, or one group of fixed_rows rows when counts
// is NULL) are cut into 128-row m-tiles.  mt_info[m] = {group, row0, nrows,
// group first row}; group_mt_begin[g] = first m-tile of group g (n_groups + 1
// entries, the last being the total).  offsets_out (nullable) receives the
// exclusive prefix of the group row counts.
constexpr int kMTile = 128;
inline int max_mtiles(long long rows, int n_groups) {
  return static_cast<int>((rows + kMTile - 1) / kMTile) + n_groups;
}
// Row counts per group come from `counts`, else from `offsets_in` (n_groups+1
// entries), else each group has fixed_rows rows.
cudaError_t launch_build_mtiles(const int32_t* counts, const int32_t* offsets_in, int fixed_rows,
                                int n_groups, int32_t* offsets_out, int4* mt_info,
                                int32_t* group_mt_begin, cudaStream_t stream);

// ------------------------------------------------------------------ tcgen05 grouped GEMM
struct TcGemmArgs {
  const int4* mt_info;
  const int32_t* group_mt_begin;
  int n_groups;
  // pair kernel (kSwiGLU, kStore): the groups' rows straight from their offsets
  // [n_groups + 1] or, when fixed_rows > 0, fixed_rows rows each from row 0; else from
  // mt_info / group_mt_begin
  const int32_t* group_off;
  int fixed_rows;
  const int2* tile_list;  // kSimBits only
  const int32_t* n_list;  // kSimBits only
  int n_ntiles;
  int n_kblocks;
  // pair kernel: units (pair or tail tiles) per block of the tile walk; a block sweeps every
  // N tile with its units fastest (0 = the default, 8)
  int unit_group;
  // pair kernel (kSwiGLU, kStore): every group is a tail of at most 128 rows (a batch of at
  // most 128 tokens), so the ring takes the tails-only layout (four stages); offsets that
  // break this are refused (MOE_ERR_DEVICE_INDEX, no tile runs)
  int tails_only;
  int kb_per_slice;  // K blocks per B slice (the shared down projection spans slices along K)
  int nt_per_slice;  // N tiles per B slice (the shared gate/up projection spans slices along N)
  int b_up_offset;   // kSwiGLU: row of the first up-projection row inside a B slice (= H)
  __nv_bfloat16* out;
  long long ld_out;
  const int32_t* out_rowmap;  // kStore: output row = out_rowmap[row], or row when NULL
  // kSimBits
  const float* norm;                   // [rows] L2 norm of each row (fp32)
  const unsigned long long* row_hash;  // [rows] hash of each row's bits
  const __nv_bfloat16* rows;           // the rows themselves (exact-duplicate check)
  int d;
  const int32_t* bucket_off;  // [E+1]
  const long long* bits_base;  // [E] first word of bucket e's bit matrix
  unsigned* bits;
  float tau;
  // kSimBits with history: 0 none; 1 record the classes (cos >= s1 similar, <= s2
  // dissimilar) into hplanes (bits layout; x = known, y = similar); 2 also merge the classes
  // the history lookup already wrote there: a pair with a class keeps it and decides its bit
  int hist_mode;
  uint2* hplanes;
  float s1, s2;
  // kSimBits: earliest similar earlier row of each row (local index), lowered by atomicMin
  // from every tile (kNoHit: none yet)
  int32_t* first;
  unsigned* status;
  // kRouter: D = x . [W1|W2|W3] over a K range of 3*d (the three bf16 terms of W_r)
  int router_n;        // N of the MMA = E rounded up to 32
  int router_kbd;      // K blocks per term (d / 64)
  // 1: the three terms side by side along N (B = [W1; W2; W3], 3 router_n rows): each x K
  // block is loaded once, K runs over d, and the epilogue adds the three accumulators
  int router_stacked;
  int n_rows;          // T
  float* part;         // [n_ntiles (K splits)][T][router_n] fp32 partial logits
};
enum TcMode { kTcSwiGLU = 0, kTcStore = 1, kTcSimBits = 2, kTcRouter = 3 };
// A: [a_rows, K] bf16 row-major.  B: [b_slices, b_rows, b_cols] bf16 (b_cols = K per slice).
cudaError_t tc_gemm(int mode, const void* A, long long a_rows, int K, const void* B, int b_slices,
                    int b_rows, int b_cols, const TcGemmArgs& args, int grid, cudaStream_t stream);
constexpr int kTcTileN = 256;
// half the largest tail a tails-only pair launch takes (tails of at most 128 rows)
constexpr int kTailOnlyRows = 64;
constexpr int kTcTileK = 64;

// ------------------------------------------------------------------ backward GEMMs (gemm_bwd.cu)
// Rows in the padded slot space (each group's rows start at a multiple of 64,
// pad rows zero).  See gemm_bwd.cu for the four products.
enum BwdMode { kBwdDH = 0, kBwdDX = 1, kBwdDWD = 2, kBwdDWGU = 3 };
struct BwdArgs {
  // token-row modes (kBwdDH, kBwdDX): m-tiles over the padded groups
  const int4* mt_info;
  const int32_t* group_mt_begin;
  int n_groups;        // groups (experts, or shared slices for the weight modes)
  int n_ntiles;        // N tiles of 256 columns (kBwdDH/kBwdDWD: per slice, the last may be 128)
  int n_kblocks;       // token modes: K blocks
  int n_per_slice;     // kBwdDH: hidden units per weight slice (H or H_shared)
  int nt_per_slice;    // kBwdDH: N tiles per slice, ceil(n_per_slice / 256)
  int n_cols;          // kBwdDWD: output columns per group (H or H_shared)
  int kb_per_slice;    // kBwdDX: K blocks per W_gu slice (2H / 64)
  // weight modes (kBwdDWD, kBwdDWGU)
  int n_mtiles;        // output-row tiles of 256 per group
  const int32_t* group_rows;  // [n_groups + 1] padded row offsets, or NULL: every group spans rows_shared rows from row 0
  int rows_shared;
  int a_col_stride;    // kBwdDWGU: A column offset per group (2H_shared for shared slices, 0 routed)
  int b_col0, b_col_stride;  // kBwdDWD: B column offset = b_col0 + group * b_col_stride
  // epilogue
  const __nv_bfloat16* au;  // kBwdDH: recomputed [a | u] per slice, row stride ld_au
  long long ld_au;
  __nv_bfloat16* out_bf16;  // kBwdDH: dA, row stride ld_out (= ld_au)
  float* out_f32;           // other modes
  long long ld_out;
  long long out_group_stride;  // weight modes: elements between groups' gradients
  long long out_group_rows;    // weight modes: out_group_stride / ld_out (set by bwd_gemm)
  unsigned* status;
};
struct BwdGemmOperands {
  const void* A;
  long long a_inner, a_rows;  // A as [a_rows][a_inner] bf16
  const void* B;
  long long b_inner, b_rows, b_slices;  // B as [b_slices][b_rows][b_inner] bf16
};
cudaError_t bwd_gemm(int mode, const BwdGemmOperands& op, const BwdArgs& args, int num_sms,
                     cudaStream_t stream);

// ------------------------------------------------------------------ backward support (backward.cu)
constexpr int kBwdPad = 64;  // group rows start at multiples of this in the padded slot space
cudaError_t launch_pad_counts(const int32_t* counts, int E, int32_t* pcounts, cudaStream_t st);
cudaError_t launch_pad_rows(const void* x_perm, const int32_t* offsets, const int32_t* poffsets,
                            const int32_t* rep_of, int E, int max_rows, int d, void* x_pad,
                            void* dy_pad, cudaStream_t st);
// mem_off [P], mem_cnt [P], mem_list [P]: the slots condensed onto each representative
// slot r are mem_list[mem_off[r] .. mem_off[r] + mem_cnt[r]), ascending.
cudaError_t launch_members(const int32_t* rep_of, const int32_t* offsets, int E, int32_t* mem_off,
                           int32_t* mem_cnt, int32_t* mem_list, cudaStream_t st);
cudaError_t launch_pad_tokens(const void* src, int T, int T_pad, int d, void* dst, cudaStream_t st);
cudaError_t launch_swiglu_from_au(const void* au, const int* n_rows_dev, int rows_max, int S,
                                  int Hs, void* h, cudaStream_t st);
cudaError_t launch_combine_bwd(const void* d_out, const void* y_pad, const int32_t* topk_idx,
                               const int32_t* slot_of, const int32_t* offsets,
                               const int32_t* poffsets, const float* gate, int T, int d, int k,
                               void* dy_pad, float* dg, cudaStream_t st);
cudaError_t launch_router_bwd(const float* logits, const int32_t* topk_idx, const float* gate,
                              const float* dg, int T, int E, int k, int gating, float* dl,
                              cudaStream_t st);
size_t router_bwd_scratch_bytes(int T, int d, int E);
cudaError_t launch_router_param_grads(const void* x, const float* dl, const float* W_r, int T,
                                      int d, int E, float* dW_r, float* d_bias, float* dx_router,
                                      void* scratch, cudaStream_t st);
cudaError_t launch_dx_assemble(const void* d_out, int add_dout, const float* dx_router,
                               const float* dz_shared, const float* dz, const int32_t* topk_idx,
                               const int32_t* slot_of, const int32_t* offsets,
                               const int32_t* poffsets, const int32_t* rep_of,
                               const int32_t* mem_off, const int32_t* mem_cnt,
                               const int32_t* mem_list, int T, int d, int k, void* dx,
                               cudaStream_t st);

// ------------------------------------------------------------------ fp32 SIMT grouped GEMM
// Same tables and tile semantics as the tensor-core path, fp32 FMA throughout.
cudaError_t simt_gemm_swiglu(const float* A, const float* B, int b_slices, int b_rows, int K,
                             int kb_per_slice_k, int nt_per_slice, int H_total, int b_up_offset,
                             const int4* mt_info, const int32_t* group_mt_begin, int n_groups,
                             int max_mt, float* out, cudaStream_t stream);
cudaError_t simt_gemm_store(const float* A, const float* B, int b_slices, int b_rows, int K,
                            int k_per_slice, int N, const int4* mt_info,
                            const int32_t* group_mt_begin, int n_groups, int max_mt,
                            const int32_t* out_rowmap, float* out, cudaStream_t stream);

// ------------------------------------------------------------------ condensation
size_t condense_scratch_bytes(int T, int k, int E);
// stats_ready: the slots' row norms and hashes are already at condense_stats_ptrs(scratch)
// (written by the dispatch), so the row-statistics pass is skipped.
cudaError_t launch_condense(const __nv_bfloat16* x_perm, const int32_t* offsets, int T, int k, int d,
                            int E, float tau, int num_sms, int32_t* rep_of, int32_t* n_rep,
                            int32_t* n_condensed, void* scratch, unsigned* status,
                            cudaStream_t stream, bool stats_ready = false);
RowStatsOut condense_stats_ptrs(void* scratch, int T, int k, int E);
// Condensation with the previous call's pair classes (Luffy's historical similarity).
// The record layout is the one include/moe.h documents for moe_condense_hist.
constexpr int kHistMagic = 0x48697374;
struct HistView {
  int32_t* header;       // {magic, T, k, E, P}
  int32_t* offsets;      // [E+1]
  int32_t* slot_of;      // [T*k]
  long long* bits_base;  // [E]
  uint2* planes;         // [P * ceil(P/32)]: x = known (the pair has a class), y = the class
};
size_t hist_record_bytes(int T, int k, int E);
HistView hist_view(const void* base, int T, int k, int E);
struct HistArgs {
  const int32_t* perm;     // [T*k] slot -> token, this call
  const int32_t* slot_of;  // [T, k] this call
  int T, k;
  float s1, s2;
  const void* hist_in;     // nullable
  void* hist_out;
  int32_t* n_cos_tiles;    // nullable
};
cudaError_t launch_condense_hist(const __nv_bfloat16* x_perm, const int32_t* offsets, int d,
                                 int E, float tau, const HistArgs& h, int num_sms,
                                 int32_t* rep_of, int32_t* n_rep, int32_t* n_condensed,
                                 void* scratch, unsigned* status, cudaStream_t stream);
// Representative rows compacted bucket by bucket: rep_rows[c] = slot of the c-th
// representative, rep_counts[e] = representatives of bucket e.
// Per bucket e: its representatives' slots in slot order at rep_local[offsets[e] ..], and
// their count rep_counts[e].
cudaError_t launch_compact_reps(const int32_t* rep_of, const int32_t* offsets, int E,
                                int32_t* rep_local, int32_t* rep_counts, cudaStream_t stream);
// The compact representative list: rows r < rep_off[E] (rep_off = exclusive prefix of the
// counts), rep_rows[r] = slot, dst[r] = src[slot]; max_rows bounds the rows (sizes the grid).
cudaError_t launch_gather_reps(int act_dtype, const void* src, const int32_t* rep_local,
                               const int32_t* offsets, const int32_t* rep_off, int E, int max_rows,
                               int d, void* dst, int32_t* rep_rows, cudaStream_t stream);

}  // namespace moe
