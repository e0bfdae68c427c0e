// Host-visible declarations of the align, permute and combine kernels
// (align_kernels.cu).
#pragma once

#include "common.cuh"

namespace moelora {

constexpr int kAlignChunk = 256;        // entries per align CTA
constexpr int kMaxBins = 11264;         // E*(L+1) held in one CTA's shared memory (44 KB)
constexpr int kMaxExperts = 1024;

struct AlignArgs {
  // router (optional): when logits is set, the align first picks each token's
  // top-k experts from logits [T][E] (fp32) and writes them to
  // topk_ids_out / topk_w_out, which then serve as topk_ids / topk_weights
  const float* logits;
  int32_t* topk_ids_out;
  float* topk_w_out;
  // inputs
  const int32_t* topk_ids;      // [T*k]; NULL = every entry on expert 0 (E == 1, k == 1)
  const int32_t* lora_ids;      // [T]
  const float* topk_weights;    // [T*k]; NULL = weight 1
  int T, k, E, L;
  int lora_ignore;               // 1: every entry's adapter is -1 (layer without LoRA)
  int n;                        // T*k
  int nbins;                    // E*(L+1)
  int nchunks;                  // ceil(n / kAlignChunk)
  int block_m;
  int Pmax;
  // scratch
  int* chunk_hist;              // [nchunks][nbins] -> per-chunk offsets
  int* bin_of;                  // [n]
  int* rank_of;                 // [n]
  int* bin_start;               // [nbins]
  WsHeader* hdr;
  // align outputs
  int* sorted_ids;              // [Pmax], may be NULL (the forward does not read it)
  int* blk_expert;              // [Pmax / block_m], may be NULL
  int* seg_off;                 // [nbins + 1], may be NULL
  int* num_post_pad;            // [1], may be NULL
  // forward extras (NULL for the plain align)
  int* row_tok;                 // [Pmax] token of each sorted row, -1 for padding
  int* row_lora;                // [Pmax] adapter of each row, -2 for padding; may be NULL
  // 1: padding rows get row_tok = -1 (and row_lora, row_w) for the permute;
  // 0 when the rows are gathered by the align itself (nothing reads them)
  int pad_rows;
  float* row_w;                 // [Pmax] gate weight of each row, 0 for padding
  int* pos_of;                  // [n] sorted row of each entry, -1 if dropped
  // token tiles, LoRA slots and shrink items for the GEMM phases
  int tn;                       // token tile width
  int spi;                      // slots per shrink item (128 / r); 0 = no LoRA
  int sks;                      // K splits of every shrink item (>= 1)
  int grp_max;                  // tiles per L2 group of the main-item order (1..255)
  TileInfo* tiles;
  ShrinkItem* shrink;           // [shrink items * sks], the splits of an item adjacent
  int* sh_cnt;                  // [2 * shrink items] split arrivals per item and CTA of a pair
  int* slot_adapter;
  int* tile_done;
  int* act_done;                // [tiles] gate_up items done per tile (two-phase launch), or NULL
  int* gu_cnt;                  // [tiles * gu_nm] split arrivals of the K-split gate_up, or NULL
  int gu_nm;
  // 1: the single-CTA align zeroes the workspace error word before anything
  // can flag it (the call then needs no separate memset)
  int reset_err;
  // Row gather fused into the small-batch align (no router): with x set, the
  // kernel runs on several CTAs; each computes the order in its own shared
  // memory, CTA 0 alone writes the tables, and the others copy the token
  // rows, x_perm[row] = x[token of row] (hv 16-byte pieces per row).
  const uint4* x;
  uint4* x_perm;
  int hv;
  // L2 prefetch by extra CTAs of the small align (pf_ctas > 0): the weights
  // that the first GEMM phase streams first, up to pf_bytes, while the
  // tables are built.  That phase's main items take the routed experts in
  // expert order (pf_expert_bytes apart from pf_base) and each expert's
  // weight tiles m = 0, 1, ...; weight tile m is rows [m * pf_rows_per_m,
  // +pf_rows_per_m) of the pf_feat_rows feature rows, and the same rows
  // pf_up_rows further on when that is not 0 (gate_up's up rows), and its
  // first K split reads bytes [pf_seg0, pf_seg1) of each pf_row_bytes row.
  const unsigned char* pf_base;
  long long pf_expert_bytes;
  long long pf_bytes;
  long long pf_row_bytes;
  long long pf_seg0, pf_seg1;
  long long pf_up_rows;
  int pf_rows_per_m;
  int pf_feat_rows;
  int pf_n_m;
  int pf_ctas;
};

// The three align kernels; hist and scatter are skipped (return success)
// when there are no entries.  `chained`: the launch may overlap the tail of
// the preceding kernel on the stream (programmatic dependent launch).
cudaError_t launch_align_hist(const AlignArgs& a, cudaStream_t stream, bool chained);
cudaError_t launch_align_scan(const AlignArgs& a, cudaStream_t stream, bool chained);
cudaError_t launch_align_scatter(const AlignArgs& a, cudaStream_t stream, bool chained);

// Router: top-k experts of each token from logits [T][E], larger logit first
// (lower index on ties), gate weights = softmax over the chosen logits.
// One warp per token; E <= 1024, k <= 32.
constexpr int kRouteMaxE = 1024;
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t stream, bool chained);

// The same align in one single-CTA kernel, for small batches; with a.x set
// (and no router) it also gathers the token rows into x_perm on extra CTAs.
constexpr int kSmallMaxBins = 8192;
bool align_small_fits(const AlignArgs& a);
cudaError_t launch_align_small(const AlignArgs& a, cudaStream_t stream, bool chained, int num_sms);

// x_perm[p] = x[row_tok[p]] for rows with a token, p < Pmax (padding rows
// are not written).  T and err serve the bounds checks of checked builds.
cudaError_t launch_permute(const __nv_bfloat16* x, const int* row_tok, __nv_bfloat16* x_perm,
                           int Pmax, int H, int T, int* err, int num_sms, cudaStream_t stream);

// out[t] = sum_j sum_s y_pair[s][pos_of[t*k+j]] in fp32 (j ascending, then
// the K splits s in order), one bf16 rounding.  split_stride in floats.
// Pmax and err serve the bounds checks of checked builds.
cudaError_t launch_combine(const float* y_pair, const int* pos_of, __nv_bfloat16* out,
                           int T, int k, int H, int nsplit, long long split_stride, int Pmax,
                           int* err, int num_sms, cudaStream_t stream);

}  // namespace moelora
