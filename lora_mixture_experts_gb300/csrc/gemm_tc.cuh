// Host-visible declarations of the tcgen05 grouped GEMM (gemm_tc.cu).
#pragma once

#include <cuda.h>
#include "common.cuh"

namespace moelora {

enum GemmMode : int { kModeGateUp = 0, kModeDown = 1, kModeLinear = 2 };

// Tensor maps of one GEMM phase.  b[i] / z[i] load 16 << i rows.
struct alignas(64) GemmMaps {
  CUtensorMap w;      // base weights, 3D (K, rows, E); gate_up: 4D (K, I, 2, E)
  CUtensorMap lb;     // LoRA expand weights B, 4D (r, rows, E, L); gate_up: 5D (r, I, 2, E, L)
  CUtensorMap la;     // LoRA shrink weights A, 4D (K, r, E, L)
  CUtensorMap la_run; // the same with a box of 128 / r consecutive adapters
  CUtensorMap b[5];   // token operand (x_perm or act), 2D (K, rows)
  CUtensorMap z[5];   // shrink results, 2D (r, slots * tn)
};

constexpr int kMaxKSplit = 4;

struct GemmParams {
  int mode;            // GemmMode
  int K;               // base reduction length
  int n_mtiles;        // weight tiles per token tile (128 rows; 256 on CTA pairs)
  int out_feats;       // valid output features (I, H or N)
  int r;               // LoRA rank, 0 = no LoRA
  int lora_w;          // elements of one LoRA K-chunk in shared memory (<= 64)
  int lora_chunks;     // r / lora_w
  int lora_swz;        // descriptor layout code of a LoRA chunk
  int done_target;     // shrink items a tile must see done: 1x or 2x its nsh
  int ksplit;          // K splits of the main items (down mode: fp32 partial per split;
                       // gate_up: parts summed by the last split, see gu_part)
  // first K block (moe_gemm_kblock_width wide) of each split,
  // split_k0[ksplit] = K blocks in all;
  // the last split is the shortest (see split_starts on the host)
  int split_k0[kMaxKSplit + 1];
  long long split_stride;  // elements between the fp32 partials of consecutive splits
  const WsHeader* hdr;
  int* err;
  const TileInfo* tiles;
  const ShrinkItem* shrink;
  const int* slot_adapter;
  const int* row_lora;
  const int* bin_start;   // first sorted row of each (expert, adapter + 1) bin
  int lp1;                // adapter bins per expert (L + 1)
  const float* row_w;
  const int* row_tok;
  int* tile_done;
  // Shrink items split K in sh_splits parts (1 = not split).  Each split
  // writes its fp32 result to zpart [sh_splits][zpart_slots * tn][r]; the
  // split whose arrival on sh_cnt (per item and CTA of a pair) comes last
  // sums the parts in split order and writes zbuf.
  int sh_splits;
  float* zpart;
  // Two-phase launch (gate_up then down in one persistent launch): the
  // gate_up phase counts each finished item on act_count[tile]; a down item
  // waits until act_wait[tile] reaches act_target (the tile's gate_up items).
  // Both NULL in a one-phase launch.
  int* act_count;
  const int* act_wait;
  int act_target;
  // sizes for the device-side bounds checks of checked builds
  int Pmax;               // sorted-row capacity
  int T;                  // tokens
  int n_experts;
  int zpart_slots;
  int* sh_cnt;
  // Shrink results [slots * tn][z_parts * r].  z_parts = 2 keeps each as two
  // bf16 rows, hi = bf16(z) and lo = bf16(z - hi) ([hi r | lo r]), and the
  // expand multiplies both, seeing z to about 16 significant bits: used for
  // the gate_up LoRA, whose rounding error SiLU(gate) * up amplifies (a
  // single bf16 z there put outputs 6-7 RMS from zero past 3e-2 x RMS).
  // z_parts = 1: one bf16 row (down and dense linear).
  __nv_bfloat16* zbuf;
  int z_parts;
  __nv_bfloat16* out;   // act [Pmax][I] (gate_up) or out [T][N] (linear)
  float* out_f32;       // y_pair [Pmax][H] (down): gate-weighted expert output, fp32
  int out_ld;
  // gate_up split over K (ksplit > 1, single-CTA tiles): each split writes
  // its fp32 part of the item's 128 accumulator rows to gu_part
  // [ksplit][gu_slots][128][tn] (slot = tile * n_mtiles + m) and counts on
  // gu_cnt[slot] (zeroed by the align); the split that arrives last sums the
  // parts in split order and applies SiLU(gate) * up
  float* gu_part;
  int* gu_cnt;
  int gu_slots;
  int* work_ctr;        // items claimed so far (zeroed by the align); NULL = fixed shares
  int spread_shrink;    // 1: on CTA pairs, spread the shrink entries over the first K split
                        //    (set when the launch's token rows are too large to stay in L2)
  int early_weights;    // 1: on unpaired tiles, stream the first weight blocks before
                        //    the preceding launch has finished (see the kernel)
};

// Launches one GEMM phase (a tile's shrink items before its main items) as a
// persistent kernel on up to `grid` work units (CTAs, or CTA pairs for
// paired tiles), capped at what can be resident at once.  tn is 16, 32, 64,
// 128 or 256.
cudaError_t launch_moe_gemm(int tn, const GemmMaps& maps, const GemmParams& p, int grid,
                            cudaStream_t stream);

// Both phases of the layer in one persistent launch (single-CTA tiles only,
// tn < 256): the gate_up items (maps0 / p0, p0.act_count set), then the down
// items (maps1 / p1, p1.act_wait and act_target set).
cudaError_t launch_moe_gemm_two_phase(int tn, const GemmMaps& maps0, const GemmParams& p0,
                                      const GemmMaps& maps1, const GemmParams& p1, int grid,
                                      cudaStream_t stream);

// Dynamic shared memory of the kernel for a token-tile width.
size_t moe_gemm_smem_bytes(int tn);

// Whether tiles of this width run on CTA pairs (2-SM MMA): then an item
// covers 256 weight rows (gate_up: 128 features) instead of 128 (64).
bool moe_gemm_paired(int tn);

// K blocks per pipeline stage for a token-tile width.
int moe_gemm_stage_kblocks(int tn);

// Width (elements) of one K block for a token-tile width: the box width of
// the K-major tensor maps and the unit of GemmParams::split_k0.
int moe_gemm_kblock_width(int tn);

}  // namespace moelora
