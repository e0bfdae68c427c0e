// Align (group routed entries by expert and adapter), permute and combine.
//
// Align follows the grouping of the multi-LoRA MoE blog ("Implementing
// multi-LoRA for MoE in vLLM": fused_moe runs one GEMM per expert over its
// tokens and fused_moe_lora adds a grid dimension over the active adapters).
// The order is the stable sort of the entries by (expert, adapter+1), done as
// a three-kernel counting sort that needs no atomics for positions:
//   hist    -- per 256-entry chunk: bin of every entry, its rank among the
//              chunk's earlier entries of the same bin, the chunk histogram;
//   scan    -- one CTA: per-bin chunk offsets, expert counts, per-expert
//              padding to block_m, segment offsets, padding rows, and the
//              token-tile / LoRA-slot / shrink-item tables of the GEMMs;
//   scatter -- position = bin start + chunk offset + rank.
// Every position is a pure function of the inputs, so the result is
// bit-identical run to run.
#include "align.cuh"

#include <cmath>

#include <algorithm>

namespace moelora {
namespace {

constexpr int kScanThreads = 1024;

// ---------------------------------------------------------------- router
// Top-k of one token's logits by one warp: k rounds of a warp argmax (larger
// logit first, lower expert index on ties; NaN never wins), then the gate
// weights as the softmax of the chosen logits.  Lane j < k keeps expert j.
__device__ __forceinline__ void route_token(const float* __restrict__ lg, int E, int k,
                                            int32_t* __restrict__ ids, float* __restrict__ w,
                                            int lane) {
  uint32_t taken = 0;          // slot i of this lane <-> expert lane + 32 i
  int my_id = -1;
  float my_l = 0.0f;
  for (int r = 0; r < k; ++r) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
    for (int i = 0, e = lane; e < E; ++i, e += 32) {
      if (taken & (1u << i)) continue;
      const float v = lg[e];
      if (v > bv || (v == bv && e < be)) {
        bv = v;
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
    if (be != 0x7fffffff && (be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == r) {
      my_id = be == 0x7fffffff ? -1 : be;
      my_l = bv;
    }
  }
  // softmax over the chosen logits (the first pick holds the largest)
  const float m = __shfl_sync(0xffffffffu, my_l, 0);
  const float ex = (lane < k && my_id >= 0) ? expf(my_l - m) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids[lane] = my_id;
    w[lane] = ex / sum;
  }
}

constexpr int kRouteWarps = 8;

__global__ void __launch_bounds__(kRouteWarps * 32) route_kernel(const float* __restrict__ logits,
                                                                 int T, int E, int k,
                                                                 int32_t* __restrict__ ids,
                                                                 float* __restrict__ w) {
  grid_dependency_wait();
  grid_dependency_trigger();
  const int t = blockIdx.x * kRouteWarps + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token(logits + static_cast<size_t>(t) * E, E, k, ids + static_cast<size_t>(t) * k,
              w + static_cast<size_t>(t) * k, threadIdx.x & 31);
}

__global__ void __launch_bounds__(kAlignChunk) align_hist_kernel(AlignArgs a) {
  grid_dependency_wait();
  grid_dependency_trigger();
  __shared__ int bins[kAlignChunk];
  extern __shared__ int hist[];   // [nbins]
  const int c = blockIdx.x;
  const int tid = threadIdx.x;
  const int f = c * kAlignChunk + tid;
  int bin = -1;
  if (f < a.n) {
    const int e = a.topk_ids ? a.topk_ids[f] : 0;
    const int l = a.lora_ignore ? -1 : a.lora_ids[f / a.k];
    if (e < 0 || e >= a.E || l < -1 || l >= a.L)
      flag_error(&a.hdr->err, kStatusBadIndex);
    else
      bin = e * (a.L + 1) + l + 1;
  }
  bins[tid] = bin;
  for (int b = tid; b < a.nbins; b += kAlignChunk) hist[b] = 0;
  __syncthreads();
  if (bin >= 0) atomicAdd(&hist[bin], 1);
  int rank = 0;
  for (int i = 0; i < tid; ++i) rank += (bins[i] == bin);
  if (f < a.n) {
    a.bin_of[f] = bin;
    a.rank_of[f] = rank;
  }
  __syncthreads();
  int* out = a.chunk_hist + static_cast<size_t>(c) * a.nbins;
  for (int b = tid; b < a.nbins; b += kAlignChunk) out[b] = hist[b];
}

// Exclusive scan of one value per thread over the block (up to 32 warps).
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = lane < nwarps ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    warp_sums[lane] = s;   // inclusive
  }
  __syncthreads();
  const int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  if (total) *total = warp_sums[nwarps - 1];
  __syncthreads();
  return excl;
}

// Exclusive scans of three values per thread over the block at once (one
// pass: two barriers instead of six); warp_sums holds 3 x 32 ints.
__device__ void block_exclusive_scan3(int v0, int v1, int v2, int* warp_sums, int& e0, int& e1, int& e2,
                                      int& t0, int& t1, int& t2) {
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int nwarps = (blockDim.x + 31) >> 5;
  int x0 = v0, x1 = v1, x2 = v2;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y0 = __shfl_up_sync(0xffffffffu, x0, o);
    const int y1 = __shfl_up_sync(0xffffffffu, x1, o);
    const int y2 = __shfl_up_sync(0xffffffffu, x2, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
      x2 += y2;
    }
  }
  if (lane == 31) {
    warp_sums[warp] = x0;
    warp_sums[32 + warp] = x1;
    warp_sums[64 + warp] = x2;
  }
  __syncthreads();
  // the second level: series q by warp q % nwarps (a block may have fewer
  // than three warps)
  for (int q = warp; q < 3; q += nwarps) {
    int v = lane < nwarps ? warp_sums[32 * q + lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_sums[32 * q + lane] = v;   // inclusive
  }
  __syncthreads();
  e0 = x0 - v0 + (warp > 0 ? warp_sums[warp - 1] : 0);
  e1 = x1 - v1 + (warp > 0 ? warp_sums[32 + warp - 1] : 0);
  e2 = x2 - v2 + (warp > 0 ? warp_sums[64 + warp - 1] : 0);
  t0 = warp_sums[nwarps - 1];
  t1 = warp_sums[32 + nwarps - 1];
  t2 = warp_sums[64 + nwarps - 1];
  __syncthreads();
}

// Everything after the per-bin totals: expert counts and padding, segment
// offsets, padding rows, block experts, and the GEMM tables.  `sb` is a
// shared-memory array holding the per-bin entry counts; it is turned into
// bin starts there (and copied to a.bin_start).  Reading the bins from shared
// memory keeps the per-expert loops free of global round trips.  Run by all
// threads of one CTA (at least one per expert).
// With write == false (the extra CTAs of the fused small align) only the bin
// starts in sb are computed; nothing is written to global memory.
__device__ void align_tables(const AlignArgs& a, int* warp_sums, int* sb, bool write = true) {
  const int tid = threadIdx.x;
  const int Lp = a.L + 1;
  // one expert per thread
  const int e = tid;
  const bool has_e = e < a.E;
  int cnt = 0;
  if (has_e)
    for (int l = 0; l < Lp; ++l) cnt += sb[e * Lp + l];
  const int pad = has_e ? (cnt + a.block_m - 1) / a.block_m * a.block_m : 0;
  int P;
  const int start = block_exclusive_scan(pad, warp_sums, &P);
  // every thread read its own expert's totals above; each overwrites only its own bins

  if (has_e) {
    int s = start;
    for (int l = 0; l < Lp; ++l) {
      const int b = e * Lp + l;
      const int tot = sb[b];
      sb[b] = s;
      if (write) {
        a.bin_start[b] = s;
        if (a.seg_off) a.seg_off[b] = s;
      }
      s += tot;
    }
  }
  if (!write) return;
  // padding and unused rows: the sentinel in sorted_ids (align entry point),
  // and no token for the permute when it runs (the forward's own tables skip
  // what nothing reads)
  const bool pad_tok = a.row_tok != nullptr && a.pad_rows;
  if (has_e) {
    if (a.blk_expert)
      for (int blk = start / a.block_m; blk < (start + pad) / a.block_m; ++blk) a.blk_expert[blk] = e;
    if (a.sorted_ids || pad_tok) {
      for (int p = start + cnt; p < start + pad; ++p) {
        if (a.sorted_ids) a.sorted_ids[p] = a.n;
        if (pad_tok) {
          a.row_tok[p] = -1;
          if (a.row_lora) a.row_lora[p] = -2;
          a.row_w[p] = 0.0f;
        }
      }
    }
  }
  if (a.sorted_ids || pad_tok) {
    for (int p = P + tid; p < a.Pmax; p += blockDim.x) {
      if (a.sorted_ids) a.sorted_ids[p] = a.n;
      if (pad_tok) {
        a.row_tok[p] = -1;
        if (a.row_lora) a.row_lora[p] = -2;
        a.row_w[p] = 0.0f;
      }
    }
  }
  if (a.blk_expert)
    for (int blk = P / a.block_m + tid; blk < a.Pmax / a.block_m; blk += blockDim.x)
      a.blk_expert[blk] = -1;
  if (tid == 0) {
    if (a.seg_off) a.seg_off[a.nbins] = P;
    if (a.num_post_pad) *a.num_post_pad = P;
    a.hdr->P = P;
  }
  if (!a.tiles) return;   // plain align: no GEMM tables

  // token tiles of tn rows per expert; one LoRA slot per adapter (>= 0)
  // present in a tile; shrink items of up to spi slots
  __shared__ int s_nh_max;   // most shrink items of any one tile
  if (tid == 0) s_nh_max = 0;
  __syncthreads();
  int n_t = 0, n_s = 0, n_h = 0, nh_max = 0;
  if (has_e && cnt > 0) {
    n_t = (cnt + a.tn - 1) / a.tn;
    if (a.spi > 0) {
      for (int j = 0; j < n_t; ++j) {
        const int s0 = start + j * a.tn;
        const int s1 = min(start + cnt, s0 + a.tn);
        int ns = 0;
        for (int l = 1; l < Lp; ++l) {
          const int lo = sb[e * Lp + l];
          const int hi = (l + 1 < Lp) ? sb[e * Lp + l + 1] : start + cnt;
          if (lo < hi && lo < s1 && hi > s0) ++ns;
        }
        n_s += ns;
        n_h += (ns + a.spi - 1) / a.spi;
        nh_max = max(nh_max, (ns + a.spi - 1) / a.spi);
      }
    }
  }
  if (nh_max > 0) atomicMax(&s_nh_max, nh_max);
  int tot_t, tot_s, tot_h, tbase, sbase, hbase;
  block_exclusive_scan3(n_t, n_s, n_h, warp_sums, tbase, sbase, hbase, tot_t, tot_s, tot_h);
  if (a.gu_cnt)   // the K-split gate_up's arrival counters, one per (tile, weight tile)
    for (int i = tid; i < tot_t * a.gu_nm; i += blockDim.x) a.gu_cnt[i] = 0;
  const int gmax = min(255, max(1, a.grp_max));
  if (has_e && cnt > 0) {
    int sl = sbase, sh = hbase;
    for (int j = 0; j < n_t; ++j) {
      const int s0 = start + j * a.tn;
      const int s1 = min(start + cnt, s0 + a.tn);
      TileInfo ti;
      ti.expert = e;
      ti.row0 = s0;
      ti.nrows = s1 - s0;
      ti.slot_base = sl;
      ti.sh_base = sh * a.sks;
      {
        // the expert's tiles in runs of at most gmax (the last run takes the rest)
        const int g0 = j / gmax * gmax;
        ti.grp = ((tbase + g0) << 8) | min(gmax, n_t - g0);
      }
      int ns = 0;
      if (a.spi > 0) {
        for (int l = 1; l < Lp; ++l) {
          const int lo = sb[e * Lp + l];
          const int hi = (l + 1 < Lp) ? sb[e * Lp + l + 1] : start + cnt;
          if (lo < hi && lo < s1 && hi > s0) a.slot_adapter[sl + ns++] = l - 1;
        }
      }
      ti.nslots = ns;
      const int nh = a.spi > 0 ? (ns + a.spi - 1) / a.spi : 0;
      ti.nsh = nh;
      for (int h = 0; h < nh; ++h) {
        ShrinkItem si;
        si.tile = tbase + j;
        si.slot0 = sl + h * a.spi;
        si.nslot = min(a.spi, ns - h * a.spi);
        for (int s = 0; s < a.sks; ++s) {
          si.ks = s;
          a.shrink[(sh + h) * a.sks + s] = si;
        }
        a.sh_cnt[2 * (sh + h)] = 0;
        a.sh_cnt[2 * (sh + h) + 1] = 0;
      }
      a.tiles[tbase + j] = ti;
      a.tile_done[tbase + j] = 0;
      if (a.act_done) a.act_done[tbase + j] = 0;
      sl += ns;
      sh += nh;
    }
  }
  if (tid == 0) {
    a.hdr->n_tiles = tot_t;
    a.hdr->n_slots = tot_s;
    a.hdr->n_shrink = tot_h * a.sks;
    a.hdr->sh_max = s_nh_max * a.sks;   // (the scan above ended with a barrier)
    a.hdr->work[0] = 0;
    a.hdr->work[1] = 0;
  }
}

__global__ void __launch_bounds__(kScanThreads) align_scan_kernel(AlignArgs a) {
  __shared__ int warp_sums[96];
  extern __shared__ int sb[];   // [nbins]
  grid_dependency_wait();
  grid_dependency_trigger();
  const int tid = threadIdx.x;

  // per-bin chunk offsets (in place) and totals; chunks are read eight at a
  // time so the loads of a bin are in flight together
  for (int b = tid; b < a.nbins; b += kScanThreads) {
    int run = 0;
    for (int c0 = 0; c0 < a.nchunks; c0 += 8) {
      int v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        v[u] = c0 + u < a.nchunks ? a.chunk_hist[static_cast<size_t>(c0 + u) * a.nbins + b] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < a.nchunks) {
          a.chunk_hist[static_cast<size_t>(c0 + u) * a.nbins + b] = run;
          run += v[u];
        }
      }
    }
    sb[b] = run;
  }
  __syncthreads();
  align_tables(a, warp_sums, sb);
}

// Bulk prefetch of [p, p + bytes) into L2 (p and bytes 16-byte multiples).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

// Weight prefetch of the small align: CTA pi of n_pf flags the experts that
// have entries, ranks them in expert order (the order of their token tiles,
// and so of the first GEMM phase's main items), and issues its share of L2
// prefetches of what that phase reads first: whole experts in 64 KB pieces
// when it does not split K, else the first split's slice of each weight
// row, weight tile by weight tile, up to pf_bytes.  The copies run in the
// memory system while the align's other CTAs build the tables, so the GEMM's
// first items read them from L2 instead of HBM, which the align leaves
// idle.  Nothing is written; the CTA returns.
__device__ void align_prefetch(const AlignArgs& a, int* warp_sums, int* cnt, int pi, int n_pf) {
  __shared__ int s_list[8];   // routed experts, in order, whose bytes are prefetched
  const int tid = threadIdx.x;
  for (int e = tid; e < a.E; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  for (int f = tid; f < a.n; f += blockDim.x) {
    const int e = a.topk_ids ? a.topk_ids[f] : 0;
    if (e >= 0 && e < a.E) cnt[e] = 1;   // (a flag: any entry makes the expert routed)
  }
  __syncthreads();
  const bool routed = tid < a.E && cnt[tid] > 0;
  int n_routed;
  const int rank = block_exclusive_scan(routed ? 1 : 0, warp_sums, &n_routed);
  const long long eb = a.pf_expert_bytes;
  const long long seg = a.pf_seg1 - a.pf_seg0;
  const bool whole = a.pf_seg0 == 0 && seg == a.pf_row_bytes;
  const int rpt = a.pf_rows_per_m * (a.pf_up_rows ? 2 : 1);   // rows per weight tile
  const long long per_expert = static_cast<long long>(a.pf_n_m) * rpt;
  const long long want = whole ? (a.pf_bytes + eb - 1) / eb : (a.pf_bytes / seg + per_expert - 1) / per_expert;
  const int n_list = static_cast<int>(min(static_cast<long long>(min(n_routed, 8)), want));
  if (routed && rank < n_list) s_list[rank] = tid;
  __syncthreads();
  if (whole) {
    const long long total = min(a.pf_bytes, n_list * eb) & ~15ll;
    constexpr long long kChunk = 1 << 16;
    const long long n_chunks = (total + kChunk - 1) / kChunk;
    for (long long c = pi + static_cast<long long>(n_pf) * tid; c < n_chunks;
         c += static_cast<long long>(n_pf) * blockDim.x) {
      const long long off = c * kChunk;
      const int li = static_cast<int>(off / eb);
      const long long o = off - li * eb;
      const long long bytes = min(min(kChunk, eb - o), total - off);
      if (bytes >= 16)
        prefetch_l2_bulk(a.pf_base + static_cast<long long>(s_list[li]) * eb + o,
                         static_cast<uint32_t>(bytes & ~15ll));
    }
    return;
  }
  const long long units = min(a.pf_bytes / seg, n_list * per_expert);
  for (long long u = pi + static_cast<long long>(n_pf) * tid; u < units;
       u += static_cast<long long>(n_pf) * blockDim.x) {
    const int li = static_cast<int>(u / per_expert);
    const long long rem = u - li * per_expert;
    const int m = static_cast<int>(rem / rpt);
    const int q = static_cast<int>(rem - static_cast<long long>(m) * rpt);
    const int fr = m * a.pf_rows_per_m + (q < a.pf_rows_per_m ? q : q - a.pf_rows_per_m);
    if (fr >= a.pf_feat_rows) continue;
    const long long row = fr + (q < a.pf_rows_per_m ? 0 : a.pf_up_rows);
    prefetch_l2_bulk(a.pf_base + static_cast<long long>(s_list[li]) * eb + row * a.pf_row_bytes + a.pf_seg0,
                     static_cast<uint32_t>(seg));
  }
}

// The whole align in one CTA for up to kScanThreads entries (decode-sized
// batches), launched with max(entries, experts) threads rounded to a warp:
// bins, stable in-bin ranks (the warps holding entries take turns in entry
// order, a warp's lanes are ordered among themselves), totals, the shared
// tables step, then the scatter.  Same results as hist + scan + scatter.
// (one CTA per SM is all it ever needs: with the default register budget for
// 1024-thread CTAs the compiler spilled; 48 registers, no spills, measured
// decode 238.9 -> 238.4 us and dense T = 1 86.7 -> 85.7 us)
__global__ void __launch_bounds__(kScanThreads, 1) align_small_kernel(AlignArgs a) {
  __shared__ int warp_sums[96];
  extern __shared__ int sm_bins[];   // [nbins] running counts, then [n] positions (gather)
  // The last pf_ctas CTAs prefetch weights into L2 (no router here: the ids
  // are inputs).  A prefetch writes nothing and L2 is coherent, so they do
  // not wait for the preceding kernel: ids read before it has finished can
  // at worst aim the prefetch at the wrong weights (ids out of range are
  // skipped), and starting during the preceding kernel gives the copies more
  // of the time the HBM would sit idle.
  const int n_pf = a.pf_ctas > 0 && a.pf_base && !a.logits ? a.pf_ctas : 0;
  if (static_cast<int>(blockIdx.x) >= static_cast<int>(gridDim.x) - n_pf) {
    align_prefetch(a, warp_sums, sm_bins, static_cast<int>(blockIdx.x) - (static_cast<int>(gridDim.x) - n_pf),
                   n_pf);
    return;
  }
  grid_dependency_wait();
  grid_dependency_trigger();
  const int tid = threadIdx.x;
  // CTA 0 writes the tables and flags bad ids; with the fused row gather the
  // other CTAs recompute the same order and copy rows
  const bool tables = blockIdx.x == 0;
  const bool gather = a.x != nullptr;
  if (a.reset_err && tables) {   // the call's first kernel clears the error word itself
    if (tid == 0) a.hdr->err = 0;
    __syncthreads();
  }
  const int gx = static_cast<int>(gridDim.x) - n_pf;   // the table and copying CTAs
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int f = tid;
  if (a.logits) {
    // router fused in: the CTA's warps pick every token's top-k first
    for (int t = warp; t < a.T; t += blockDim.x >> 5)
      route_token(a.logits + static_cast<size_t>(t) * a.E, a.E, a.k,
                  a.topk_ids_out + static_cast<size_t>(t) * a.k,
                  a.topk_w_out + static_cast<size_t>(t) * a.k, lane);
    __syncthreads();
  }
  int bin = -1;
  float wgt = 1.0f;
  if (f < a.n) {
    const int e = a.topk_ids ? a.topk_ids[f] : 0;
    const int l = a.lora_ignore ? -1 : a.lora_ids[f / a.k];
    if (tables && a.topk_weights) wgt = a.topk_weights[f];   // (loaded with the ids)
    if (e < 0 || e >= a.E || l < -1 || l >= a.L) {
      if (tables) flag_error(&a.hdr->err, kStatusBadIndex);
    } else {
      bin = e * (a.L + 1) + l + 1;
    }
  }
  for (int b = tid; b < a.nbins; b += blockDim.x) sm_bins[b] = 0;
  __syncthreads();
  int rank = 0;
  const int entry_warps = (a.n + 31) >> 5;
  for (int w = 0; w < entry_warps; ++w) {
    if (warp == w) {
      const unsigned peers = __match_any_sync(0xffffffffu, bin);
      const int leader = __ffs(peers) - 1;
      if (bin >= 0) rank = sm_bins[bin] + __popc(peers & ((1u << lane) - 1));
      __syncwarp();
      if (bin >= 0 && lane == leader) sm_bins[bin] += __popc(peers);
    }
    __syncthreads();
  }
  align_tables(a, warp_sums, sm_bins, tables);
  __syncthreads();
  int* sm_pos = sm_bins + a.nbins;
  if (f < a.n) {
    const int pos = bin < 0 ? -1 : sm_bins[bin] + rank;
    if (gather) sm_pos[f] = pos;
    if (tables) {
      if (bin < 0 || !MOELORA_IN_RANGE(&a.hdr->err, pos, 0, a.Pmax)) {
        if (a.pos_of) a.pos_of[f] = -1;
      } else {
        if (a.sorted_ids) a.sorted_ids[pos] = f;
        if (a.row_tok) {
          a.row_tok[pos] = f / a.k;
          if (a.row_lora) a.row_lora[pos] = bin % (a.L + 1) - 1;
          a.row_w[pos] = wgt;
          a.pos_of[f] = pos;
        }
      }
    }
  }
  if (gather && (gx == 1 || !tables)) {
    // rows of the entries, 16-byte pieces spread over the copying CTAs
    // (CTAs 1.. when there are several); padding rows are not written
    __syncthreads();
    const int copiers = gx > 1 ? gx - 1 : 1;
    const int ci = gx > 1 ? static_cast<int>(blockIdx.x) - 1 : 0;
    // (a thread's pieces are loaded together, then stored: four row reads in
    // flight instead of one after another; on the decode batch the copying
    // CTAs' row copy took 3.1 us, now 1.7 us, and the call 238.2 -> 237.1 us)
    const long long total = static_cast<long long>(a.n) * a.hv;
    const long long stride = static_cast<long long>(copiers) * blockDim.x;
    constexpr int kBatch = 4;
    for (long long i0 = static_cast<long long>(ci) * blockDim.x + tid; i0 < total; i0 += kBatch * stride) {
      uint4 v[kBatch];
      long long dst[kBatch];
#pragma unroll
      for (int q = 0; q < kBatch; ++q) {
        const long long i = i0 + q * stride;
        dst[q] = -1;
        if (i < total) {
          const int fe = static_cast<int>(i / a.hv);
          const int u = static_cast<int>(i - static_cast<long long>(fe) * a.hv);
          const int pos = sm_pos[fe];
          if (pos >= 0 && MOELORA_IN_RANGE(&a.hdr->err, pos, 0, a.Pmax)) {
            v[q] = a.x[static_cast<size_t>(fe / a.k) * a.hv + u];
            dst[q] = static_cast<long long>(pos) * a.hv + u;
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kBatch; ++q)
        if (dst[q] >= 0) a.x_perm[dst[q]] = v[q];
    }
  }
}

__global__ void __launch_bounds__(kAlignChunk) align_scatter_kernel(AlignArgs a) {
  grid_dependency_wait();
  grid_dependency_trigger();
  const int c = blockIdx.x;
  const int f = c * kAlignChunk + threadIdx.x;
  if (f >= a.n) return;
  const int bin = a.bin_of[f];
  if (bin < 0) {
    if (a.pos_of) a.pos_of[f] = -1;
    return;
  }
  const int pos = a.bin_start[bin] + a.chunk_hist[static_cast<size_t>(c) * a.nbins + bin] +
                  a.rank_of[f];
  if (!MOELORA_IN_RANGE(&a.hdr->err, pos, 0, a.Pmax)) {
    if (a.pos_of) a.pos_of[f] = -1;
    return;
  }
  if (a.sorted_ids) a.sorted_ids[pos] = f;
  if (a.row_tok) {
    a.row_tok[pos] = f / a.k;
    if (a.row_lora) a.row_lora[pos] = bin % (a.L + 1) - 1;
    a.row_w[pos] = a.topk_weights ? a.topk_weights[f] : 1.0f;
    a.pos_of[f] = pos;
  }
}

// One warp per (sorted row, chunk of 32 * kPermUnroll 16-byte pieces): the
// row's token is read once and the lane's pieces are copied with all their
// loads in flight.  Rows without a token (the per-expert padding and the
// rows past the padded total) are not written: a tile reads them only into
// MMA columns that its epilogue drops, and each D column depends on its own
// token row alone.
constexpr int kPermUnroll = 4;

__global__ void __launch_bounds__(256) permute_kernel(const uint4* __restrict__ x,
                                                      const int* __restrict__ row_tok,
                                                      uint4* __restrict__ x_perm, int Pmax, int hv,
                                                      int T, int* err) {
  grid_dependency_wait();
  grid_dependency_trigger();
  const int lane = threadIdx.x & 31;
  const int per_row = (hv + 32 * kPermUnroll - 1) / (32 * kPermUnroll);
  const long long items = static_cast<long long>(Pmax) * per_row;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5); w < items;
       w += nw) {
    const int p = static_cast<int>(w / per_row);
    const int c0 = static_cast<int>(w - static_cast<long long>(p) * per_row) * 32 * kPermUnroll + lane;
    const int t = row_tok[p];
    if (t < 0 || !MOELORA_IN_RANGE(err, t, 0, T)) continue;
    const uint4* src = x + static_cast<size_t>(t) * hv;
    uint4* dst = x_perm + static_cast<size_t>(p) * hv;
    uint4 v[kPermUnroll];
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < hv) v[u] = __ldg(src + c);
    }
#pragma unroll
    for (int u = 0; u < kPermUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c < hv) dst[c] = v[u];
    }
  }
}

// out[t] = sum over the token's k pairs (j ascending) and, inside a pair, its
// K-split partials (split ascending) of the fp32 rows y_pair[pos_of[t, j]],
// rounded once to bf16.  One warp per (token, chunk of 32 * kCombUnroll
// four-feature groups): the token's positions are read once, then all
// K x NS x kCombUnroll partial loads of a lane are in flight together.  The
// summation order is fixed, so the result is deterministic.
constexpr int kCombUnroll = 2;

template <int K, int NS>
__global__ void __launch_bounds__(128) combine_kernel(const float4* __restrict__ y_pair,
                                                      const int* __restrict__ pos_of,
                                                      uint2* __restrict__ out, int T, int kk,
                                                      int nsplit, int hv, long long split_stride4,
                                                      int Pmax, int* err) {
  const int k = K > 0 ? K : kk;
  const int ns = NS > 0 ? NS : nsplit;
  const int lane = threadIdx.x & 31;
  const int per_tok = (hv + 32 * kCombUnroll - 1) / (32 * kCombUnroll);
  const long long items = static_cast<long long>(T) * per_tok;
  const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  const long long w0 = blockIdx.x * static_cast<long long>(blockDim.x >> 5) + (threadIdx.x >> 5);
  // the rows of the warp's first token come from the align, which completed
  // before the preceding launch let this one start: read them before waiting
  // for the partial rows themselves
  int pos0[K > 0 ? K : 1];
  if (K > 0 && w0 < items) {
    const int t0 = static_cast<int>(w0 / per_tok);
#pragma unroll
    for (int j = 0; j < (K > 0 ? K : 1); ++j) pos0[j] = pos_of[static_cast<size_t>(t0) * K + j];
  }
  grid_dependency_wait();
  grid_dependency_trigger();
  for (long long w = w0; w < items; w += nw) {
    const int t = static_cast<int>(w / per_tok);
    const int c0 = static_cast<int>(w - static_cast<long long>(t) * per_tok) * 32 * kCombUnroll + lane;
    float4 acc[kCombUnroll];
#pragma unroll
    for (int u = 0; u < kCombUnroll; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (K > 0 && NS > 0) {
      int pos[K > 0 ? K : 1];
#pragma unroll
      for (int j = 0; j < K; ++j) {
        pos[j] = w == w0 ? pos0[j] : pos_of[static_cast<size_t>(t) * K + j];
        if (pos[j] >= 0 && !MOELORA_IN_RANGE(err, pos[j], 0, Pmax)) pos[j] = -1;
      }
      float4 v[K > 0 ? K : 1][NS > 0 ? NS : 1][kCombUnroll];
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int s = 0; s < NS; ++s)
#pragma unroll
          for (int u = 0; u < kCombUnroll; ++u) {
            const int c = c0 + u * 32;
            v[j][s][u] = (pos[j] >= 0 && c < hv)
                             ? y_pair[s * split_stride4 + static_cast<size_t>(pos[j]) * hv + c]
                             : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
      for (int j = 0; j < K; ++j)
#pragma unroll
        for (int s = 0; s < NS; ++s)
#pragma unroll
          for (int u = 0; u < kCombUnroll; ++u) {
            acc[u].x += v[j][s][u].x;
            acc[u].y += v[j][s][u].y;
            acc[u].z += v[j][s][u].z;
            acc[u].w += v[j][s][u].w;
          }
    } else {
      for (int j = 0; j < k; ++j) {
        const int pos = pos_of[static_cast<size_t>(t) * k + j];
        if (pos < 0 || !MOELORA_IN_RANGE(err, pos, 0, Pmax)) continue;
        for (int s = 0; s < ns; ++s)
#pragma unroll
          for (int u = 0; u < kCombUnroll; ++u) {
            const int c = c0 + u * 32;
            if (c >= hv) continue;
            const float4 v = y_pair[s * split_stride4 + static_cast<size_t>(pos) * hv + c];
            acc[u].x += v.x;
            acc[u].y += v.y;
            acc[u].z += v.z;
            acc[u].w += v.w;
          }
      }
    }
#pragma unroll
    for (int u = 0; u < kCombUnroll; ++u) {
      const int c = c0 + u * 32;
      if (c >= hv) continue;
      uint2 o;
      __nv_bfloat162* o2 = reinterpret_cast<__nv_bfloat162*>(&o);
      o2[0] = __floats2bfloat162_rn(acc[u].x, acc[u].y);
      o2[1] = __floats2bfloat162_rn(acc[u].z, acc[u].w);
      out[static_cast<size_t>(t) * hv + c] = o;
    }
  }
}

}  // namespace

cudaError_t launch_align_hist(const AlignArgs& a, cudaStream_t stream, bool chained) {
  if (a.nchunks == 0) return cudaSuccess;
  return launch_chained(align_hist_kernel, dim3(a.nchunks), dim3(kAlignChunk),
                        a.nbins * sizeof(int), stream, chained, a);
}

cudaError_t launch_align_scan(const AlignArgs& a, cudaStream_t stream, bool chained) {
  return launch_chained(align_scan_kernel, dim3(1), dim3(kScanThreads), a.nbins * sizeof(int),
                        stream, chained, a);
}

bool align_small_fits(const AlignArgs& a) {
  return a.n <= kScanThreads && a.nbins <= kSmallMaxBins && a.E <= kScanThreads;
}

cudaError_t launch_align_small(const AlignArgs& a, cudaStream_t stream, bool chained, int num_sms) {
  const int threads = (std::max(std::max(a.n, a.E), 32) + 31) / 32 * 32;
  const bool gather = a.x != nullptr && a.logits == nullptr;
  AlignArgs b = a;
  if (!gather) {
    b.x = nullptr;
    b.x_perm = nullptr;
  }
  int grid = 1;
  if (gather) {   // one table CTA plus copiers of about four pieces per thread
    const long long pieces = static_cast<long long>(a.n) * a.hv;
    grid = 1 + static_cast<int>(std::min<long long>((pieces + 4LL * threads - 1) / (4LL * threads),
                                                    std::max(1, num_sms - 1)));
  }
  if (a.pf_ctas > 0 && a.pf_base && !a.logits) grid += a.pf_ctas;   // the prefetching CTAs
  const size_t smem = (static_cast<size_t>(a.nbins) + (gather ? a.n : 0)) * sizeof(int);
  return launch_chained(align_small_kernel, dim3(grid), dim3(threads), smem, stream, chained, b);
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t stream, bool chained) {
  const int grid = std::max(1, (T + kRouteWarps - 1) / kRouteWarps);
  return launch_chained(route_kernel, dim3(grid), dim3(kRouteWarps * 32), 0, stream, chained, logits,
                        T, E, k, ids, w);
}

cudaError_t launch_align_scatter(const AlignArgs& a, cudaStream_t stream, bool chained) {
  if (a.nchunks == 0) return cudaSuccess;
  return launch_chained(align_scatter_kernel, dim3(a.nchunks), dim3(kAlignChunk), 0, stream,
                        chained, a);
}

cudaError_t launch_permute(const __nv_bfloat16* x, const int* row_tok, __nv_bfloat16* x_perm,
                           int Pmax, int H, int T, int* err, int num_sms, cudaStream_t stream) {
  const int hv = H / 8;
  const long long items =
      static_cast<long long>(Pmax) * ((hv + 32 * kPermUnroll - 1) / (32 * kPermUnroll));
  int grid = static_cast<int>(std::min<long long>((items + 7) / 8, static_cast<long long>(num_sms) * 8));
  if (grid < 1) grid = 1;
  return launch_chained(permute_kernel, dim3(grid), dim3(256), 0, stream, true,
                        reinterpret_cast<const uint4*>(x), row_tok, reinterpret_cast<uint4*>(x_perm),
                        Pmax, hv, T, err);
}

cudaError_t launch_combine(const float* y_pair, const int* pos_of, __nv_bfloat16* out,
                           int T, int k, int H, int nsplit, long long split_stride, int Pmax,
                           int* err, int num_sms, cudaStream_t stream) {
  const int hv = H / 4;
  const long long items =
      static_cast<long long>(T) * ((hv + 32 * kCombUnroll - 1) / (32 * kCombUnroll));
  int grid = static_cast<int>(std::min<long long>((items + 3) / 4, static_cast<long long>(num_sms) * 8));
  if (grid < 1) grid = 1;
  auto go = [&](auto kernel) {
    return launch_chained(kernel, dim3(grid), dim3(128), 0, stream, true,
                          reinterpret_cast<const float4*>(y_pair), pos_of, reinterpret_cast<uint2*>(out), T,
                          k, nsplit, hv, split_stride / 4, Pmax, err);
  };
  if (nsplit == 1) {
    if (k == 1) return go(combine_kernel<1, 1>);
    if (k == 2) return go(combine_kernel<2, 1>);
    if (k == 4) return go(combine_kernel<4, 1>);
    if (k == 6) return go(combine_kernel<6, 1>);
    if (k == 8) return go(combine_kernel<8, 1>);
  } else if (nsplit == 2) {
    if (k == 1) return go(combine_kernel<1, 2>);
    if (k == 2) return go(combine_kernel<2, 2>);
    if (k == 4) return go(combine_kernel<4, 2>);
    if (k == 6) return go(combine_kernel<6, 2>);
    if (k == 8) return go(combine_kernel<8, 2>);
  } else if (k == 1) {   // the dense linear's finer K splits
    if (nsplit == 3) return go(combine_kernel<1, 3>);
    if (nsplit == 4) return go(combine_kernel<1, 4>);
  }
  return go(combine_kernel<0, 0>);
}

}  // namespace moelora
