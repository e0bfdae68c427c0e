// Persistent tcgen05 grouped GEMM for the MoE-LoRA expert layer (sm_103a).
//
// One launch runs one projection phase of the layer, or on single-CTA tiles
// both (gate_up items, then down items; see gemm_body).  Per projection
// (multi-LoRA MoE blog, "Implementing multi-LoRA for MoE in vLLM": y = xW +
// xAB, the shrink z = xA and the expand zB, one GEMM per expert over its
// tokens):
//
//  * shrink items  -- z = X A[a,e]^T for the adapters present in a token tile,
//    stacked r rows per adapter in one 128-row MMA tile.  The epilogue keeps,
//    for every token, only the rows of its own adapter and writes zeros for
//    the others, so the expand can treat each adapter as one extra K-chunk.
//  * main items    -- a 128-row tile of the expert's weight rows against one
//    token tile: acc = W_tile X^T (K loop over the hidden size) followed by
//    one K-chunk of width r per adapter present: acc += B[a,e]_tile Z_a^T.
//    The epilogue applies SiLU(gate)*up (gate_up, stored bf16), the gate
//    weight (down, stored fp32 for the combine) or nothing (dense linear,
//    stored bf16).
//
// Orientation: the weight rows are the MMA's M side (128 rows) and the
// tokens its N side (16..256, rounded up to 16), so a decode-sized tile with
// a few tokens streams weights at full width and a prefill tile uses N=256.
// Operands arrive by TMA (128-byte swizzle, K-major) into a ring of shared
// memory stages; one thread issues tcgen05.mma into a double-buffered TMEM
// accumulator; four epilogue warps drain TMEM with tcgen05.ld.  A stage holds
// KB consecutive 64-wide K blocks (KB = 4 for 16-row token tiles, 2 for 32
// and 64, 1 above): at decode sizes, where the weights stream from HBM, big
// stages (64 KB of weights per barrier round trip) read markedly faster than
// 16 KB ones.  The LoRA expand chunks (r-wide, r <= 64) are packed into a
// stage by bytes: KB * 64 / r of them share one barrier round trip.
//
// 256-token tiles run on CTA pairs (2-SM MMA): the two CTAs of a cluster
// share every item, each loading its 128 weight rows and half of the token
// rows; the even CTA issues tcgen05.mma.cta_group::2 (M = 256) whose D rows
// land in both CTAs' TMEM, and both CTAs drain their own half.  Per SM this
// halves the token-operand bytes of a K block and lets a stage carry two K
// blocks (64 KB), which is what the tensor-bound prefill tiles need: TMA
// streaming from L2 measured 9 TB/s with 16 KB stages but 19-25 TB/s with 64 KB.
//
// A tile's shrink items precede its main items in the item order (all
// shrink items first, or, in large CTA-pair launches, each tile's a wave of
// items ahead of it: see ItemOrder), and a main item's producer waits
// (bounded) for its tile's shrink items before loading the z chunks.  Items
// are claimed in index order from a counter by CTAs (CTA pairs) that are
// running, so every item waited for was claimed earlier by a running CTA and
// the wait ends even when only part of the grid is resident (another
// stream's kernels holding SMs).
#include "gemm_tc.cuh"

#include <algorithm>
#include <cstddef>

namespace moelora {
namespace {

constexpr int kThreads = 224;            // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue, warp 6 items
constexpr int kSchedWarp = 6;
constexpr int kQ = 8;                    // item ring slots
constexpr int kClaimAhead = 1;           // items claimed beyond those the producer has started

// One entry of the item ring: the item index (-1 = no more items) and its
// token tile, written by the scheduling warp for the producer, MMA and
// epilogue warps of the CTA.
struct RingEntry {
  int w;
  int sh;        // shrink entry of a shrink item, -1 for a main item
  int pad_[2];
  TileInfo ti;
};
// K-block width and pipeline shape of CTA-pair tiles (the tensor-bound
// case): K blocks of MOELORA_PAIR_BK elements (64, or 32 with 64-byte rows),
// MOELORA_PAIR_KB of them per stage, MOELORA_PAIR_STAGES stages.  Measured
// on GB300 (same box): four stages of three 32-wide blocks (48 KB) against
// three of two 64-wide blocks (64 KB): prefill 805 -> 885 us, dense T = 512
// 188 -> 223 us, skewed 3.06 -> 3.28 ms; the 64-wide blocks stay.
#ifndef MOELORA_PAIR_BK
#define MOELORA_PAIR_BK 64
#endif
#ifndef MOELORA_PAIR_KB
#define MOELORA_PAIR_KB 2
#endif
#ifndef MOELORA_PAIR_STAGES
#define MOELORA_PAIR_STAGES 3
#endif

template <int TN, bool PAIR>
struct Cfg {
  // K-block width (elements): 64 (128-byte rows, 128-byte swizzle), or 32
  // on CTA pairs (64-byte rows and swizzle)
  static constexpr int kBK = PAIR ? MOELORA_PAIR_BK : 64;
  static constexpr uint32_t kSwzK = kBK == 64 ? 2u : 4u;        // descriptor layout code
  static constexpr uint32_t kSboK = 8u * kBK * 2u;                // bytes between 8-row groups
  static constexpr int kATile = 128 * kBK * 2;                    // 128 weight rows of a K block
  static constexpr int kRowsB = PAIR ? TN / 2 : TN;   // token rows a CTA holds per K block
  static constexpr int kKB =
      PAIR ? MOELORA_PAIR_KB : (TN <= 16 ? 4 : (TN <= 64 ? 2 : 1));   // K blocks per stage
  static constexpr int kBTileBytes = kRowsB * kBK * 2;             // per K block
  static constexpr int kStageBytes = kKB * (kATile + kBTileBytes);
  static constexpr int kStages =
      PAIR ? MOELORA_PAIR_STAGES : (TN <= 16 ? 3 : (TN <= 32 ? 5 : (TN <= 64 ? 4 : (TN <= 128 ? 6 : 4))));
  static constexpr int kTmemCols = 2 * TN < 32 ? 32 : 2 * TN;
  static constexpr int kBarOff = kStages * kStageBytes;
  static constexpr int kNumBars = 2 * kStages + 5 + 3 * kQ;
  static constexpr int kRingOff = kBarOff + kNumBars * 8 + 16;   // RingEntry[kQ]
  // the producer's per-stage copy accounting (4 x kStages ints), see the end
  // of gemm_body
  static constexpr int kAcctOff = kRingOff + kQ * static_cast<int>(sizeof(RingEntry));
  static constexpr int kSmemBytes = 1024 + kAcctOff + 4 * kStages * 4 + 16;
  static constexpr int kMRows = PAIR ? 256 : 128;   // weight rows of one item
  // shared-memory offset of K block j's A / B tile inside a stage
  __host__ __device__ static constexpr int a_off(int j) { return j * kATile; }
  __host__ __device__ static constexpr int b_off(int j) { return kKB * kATile + j * kBTileBytes; }
  // LoRA expand chunk j of width lw (16, 32 or 64) packed in a stage: its
  // 128 B rows in the A region, its up-to-kRowsB z rows in the B region
  // (kKB * kBK / lw chunks per stage; chunk sizes are multiples of the
  // swizzle atom, so every chunk starts on one)
  __host__ __device__ static constexpr int lora_a_off(int j, int lw) { return j * 128 * lw * 2; }
  __host__ __device__ static constexpr int lora_b_off(int j, int lw) {
    return kKB * kATile + j * kRowsB * lw * 2;
  }
};

// First K block of split s when nk blocks are cut into n splits.
__device__ __forceinline__ int split_begin(int nk, int s, int n) {
  return static_cast<int>(static_cast<long long>(nk) * s / n);
}

struct Item {
  int shrink;   // 1 = shrink item
  int tile;
  int m;        // weight tile (main items)
  int sh;       // shrink item index
  int ks;       // K split (main items)
};

// Item order of a launch phase.  Main items come K split by K split; inside
// a split, the token tiles' L2 groups in tile order.  A group is a run of
// consecutive tiles of one expert (written by the align into each tile's
// `grp`); inside it the weight tile m is the slow index and the tile the
// fast one, so the tiles of an expert read each weight tile one after the
// other while it is hot in L2, and the group's token rows (the align caps the
// run length) stay resident across all m.
//
// Shrink entries come either all first (shs == 0), or, on CTA pairs whose
// token rows exceed what L2 keeps, spread over the first split (shs > 0):
// every tile gets shs shrink slots (its shrink entries, then empty slots that
// the scheduler skips), placed `ahead` tiles before the tile itself.  The
// first split is then a prologue of the slots of tiles [0, ahead) followed by
// one block per group of tiles [g0, g0+gn): the slots of tiles [g0+ahead,
// g0+gn+ahead) (none past the last tile), then the group's main items.  A
// tile's shrink entries thus always come before its main items, about one
// wave of items earlier: they are done when the main items' expand needs
// their result, and the token rows they read are still in L2 when the main
// items read them (all shrink entries first
// made every main item re-read its rows from DRAM: +90 MB per projection on
// the prefill batch).  Since block sizes are proportional to tile counts, the
// group of a first-split item w is the group of tile (w - prologue) / (n_m +
// shs), or (later splits) of tile w / n_m: its anchor.
struct ItemOrder {
  int n_sh;      // shrink entries
  int n_tiles;
  int n_m;       // weight tiles
  int shs;       // shrink slots per tile, 0: all shrink entries first
  int ahead;     // tiles by which a tile's shrink slots precede it (shs > 0)
};

__device__ __forceinline__ void group_of(int grp, int& g0, int& gn) {
  g0 = grp >> 8;
  gn = max(1, grp & 255);
}

// Main item w of the order, given the group of its tile (any tile's `grp` in it).
__device__ __forceinline__ Item decode_main(int w, const ItemOrder& o, int grp) {
  Item it;
  int g0, gn;
  group_of(grp, g0, gn);
  const int per_split = o.n_tiles * o.n_m;
  it.shrink = 0;
  it.sh = -1;
  if (o.shs > 0) {
    const int pro = o.ahead * o.shs;
    const int region0 = pro + o.n_tiles * (o.n_m + o.shs);
    if (w < region0) {
      const int wm = w - pro - g0 * (o.n_m + o.shs) - gn * o.shs;
      it.ks = 0;
      it.m = wm / gn;
      it.tile = g0 + (wm - it.m * gn);
      return it;
    }
    w -= region0;
    it.ks = 1 + w / per_split;
    w -= (it.ks - 1) * per_split;
  } else {
    w -= o.n_sh;
    it.ks = w / per_split;
    w -= it.ks * per_split;
  }
  const int wl = w - g0 * o.n_m;
  it.m = wl / gn;
  it.tile = g0 + (wl - it.m * gn);
  return it;
}

// The scheduler's view of item w: a shrink entry (sh >= 0, tile = its tile),
// a main item (sh = -1, tile = its tile), or an empty shrink slot (false).
__device__ __forceinline__ bool resolve_item(int w, const ItemOrder& o, const TileInfo* tiles,
                                             const ShrinkItem* shrink, int sks, int& sh, int& tile) {
  const int per_split = o.n_tiles * o.n_m;
  auto slot = [&](int t, int j) -> bool {
    if (t >= o.n_tiles) return false;
    const TileInfo& ti = tiles[t];
    if (j >= ti.nsh * sks) return false;
    sh = ti.sh_base + j;
    tile = t;
    return true;
  };
  int grp;
  if (o.shs > 0) {
    const int pro = o.ahead * o.shs;
    const int region0 = pro + o.n_tiles * (o.n_m + o.shs);
    if (w < pro) return slot(w / o.shs, w % o.shs);
    if (w < region0) {
      const int w2 = w - pro;
      grp = tiles[w2 / (o.n_m + o.shs)].grp;
      int g0, gn;
      group_of(grp, g0, gn);
      const int wl = w2 - g0 * (o.n_m + o.shs);
      if (wl < gn * o.shs) return slot(g0 + wl / o.shs + o.ahead, wl % o.shs);
    } else {
      grp = tiles[((w - region0) % per_split) / o.n_m].grp;
    }
  } else {
    if (w < o.n_sh) {
      sh = w;
      tile = shrink[w].tile;
      return true;
    }
    grp = tiles[((w - o.n_sh) % per_split) / o.n_m].grp;
  }
  sh = -1;
  tile = decode_main(w, o, grp).tile;
  return true;
}

// A consumer's view of item w, from its ring entry: the shrink entry `sh`
// (spread order only; all first, shrink item w is entry w), the tile's group.
__device__ __forceinline__ Item item_of(int w, int sh, const ItemOrder& o, int grp,
                                        const ShrinkItem* shrink) {
  if (o.shs == 0) sh = w < o.n_sh ? w : -1;
  if (sh >= 0) {
    Item it;
    it.shrink = 1;
    it.sh = sh;
    it.tile = shrink[sh].tile;
    it.m = 0;
    it.ks = 0;
    return it;
  }
  return decode_main(w, o, grp);
}

// First K chunk of a main item's loop.  Concurrent items start at different
// K offsets so that their weight rows (all at the same column otherwise)
// spread over the DRAM channels instead of camping on the few that one
// column offset maps to when the row stride is a large power of two.  A pure
// function of the item: the summation order, and so the result, is the same
// on every run.
__device__ __forceinline__ int k_rotation(const Item& it, int nkc) {
  const unsigned h = static_cast<unsigned>(it.m) * 2654435761u + static_cast<unsigned>(it.tile) * 40503u +
                     static_cast<unsigned>(it.ks) * 97u;
  return static_cast<int>((h >> 7) % static_cast<unsigned>(nkc));
}

// Smallest box index i with (16 << i) >= n.
__device__ __forceinline__ int box_index(int n) {
  int i = 0;
  while ((16 << i) < n) ++i;
  return i;
}

__device__ __forceinline__ bool bar_red_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// The body of both kernels below.  A launch runs one phase (NPH = 1: maps0 /
// p0, which maps1 / p1 alias), or on single-CTA tiles both phases of the
// layer (NPH = 2: gate_up items, then down items, in one item order with one
// claim counter).  A down item of a two-phase launch waits for its token
// tile's activation rows: every gate_up main item of the tile counts on the
// tile's counter once its rows are stored.  Items are claimed in order by
// running CTAs, so the gate_up items waited for were claimed earlier by
// running CTAs and the wait ends.  NPH is a template argument so
// that the one-phase kernel reads its parameters at fixed offsets.
template <int TN, bool PAIR, int NPH, bool SPREAD>
__device__ __forceinline__ void gemm_body(const GemmMaps& maps0, const GemmMaps& maps1,
                                          const GemmParams& p0, const GemmParams& p1) {
  constexpr int n_phases = NPH;
  using C = Cfg<TN, PAIR>;
  // fields shared by the phases (tables, counters, sizes) are read from p0
  const GemmParams& p = p0;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBarOff);
  uint64_t* full_bar = bars;
  uint64_t* empty_bar = bars + C::kStages;
  uint64_t* accf_bar = bars + 2 * C::kStages;       // [2]
  uint64_t* acce_bar = bars + 2 * C::kStages + 2;   // [2]
  uint64_t* drain_bar = bars + 2 * C::kStages + 4;
  uint64_t* itemf_bar = bars + 2 * C::kStages + 5;   // [kQ] ring entry written
  uint64_t* iteme_bar = itemf_bar + kQ;              // [kQ] ring entry read by every consumer
  uint64_t* itemp_bar = iteme_bar + kQ;              // [kQ] ring entry taken by the producer
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + C::kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  RingEntry* ring = reinterpret_cast<RingEntry*>(smem + C::kRingOff);
  // Per stage slot, what the producer thread of this CTA issued into its
  // latest use (stage count, or -1, and bytes) and, on the CTA that counts a
  // stage's bytes (the leader), what it posted on the slot's full barrier.
  int* st_gen = reinterpret_cast<int*>(smem + C::kAcctOff);
  int* st_bytes = st_gen + C::kStages;
  int* po_gen = st_gen + 2 * C::kStages;
  int* po_bytes = st_gen + 3 * C::kStages;
  int* peer_abort = st_gen + 4 * C::kStages;   // the peer CTA's abort flag, copied at the end

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // CTA pairs: rank 0 leads; items are shared by the two CTAs of a cluster
  const uint32_t rank = PAIR ? cluster_rank() : 0;
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(smem_u32(&full_bar[s]), 1);
      mbar_init(smem_u32(&empty_bar[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accf_bar[b]), 1);
      mbar_init(smem_u32(&acce_bar[b]), PAIR ? 8 : 4);   // epilogue warps of both CTAs
    }
    mbar_init(smem_u32(drain_bar), 1);
    // consumers of a ring entry: producer, MMA issuer (leader only), four
    // epilogue warps; on CTA pairs the peer's five release the leader's
    // entry barrier too (the leader's scheduler writes both rings)
    for (int q = 0; q < kQ; ++q) {
      mbar_init(smem_u32(&itemf_bar[q]), 1);
      mbar_init(smem_u32(&iteme_bar[q]), PAIR ? (leader ? 11 : 1) : 6);
      mbar_init(smem_u32(&itemp_bar[q]), 1);
    }
    for (int st = 0; st < C::kStages; ++st) {
      st_gen[st] = -1;
      st_bytes[st] = 0;
      po_gen[st] = -1;
      po_bytes[st] = 0;
    }
    *peer_abort = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    for (int ph = 0; ph < n_phases; ++ph) {
      const GemmMaps& mp = NPH == 2 && ph ? maps1 : maps0;
      tma_prefetch_desc(&mp.w);
      if (p.r > 0) {
        tma_prefetch_desc(&mp.lb);
        tma_prefetch_desc(&mp.la);
        tma_prefetch_desc(&mp.la_run);
      }
    }
  }
  if (warp == 1) {
    if (PAIR)
      tmem_alloc_pair(smem_u32(tmem_holder), C::kTmemCols);
    else
      tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // the peer's barriers exist before any remote signal
  tc_fence_after();
  // Results of the preceding launch (x_perm / act) are read only after the
  // grid dependency wait; the next launch may start its own preamble.  On
  // unpaired tiles the scheduling and producer warps do not wait here: the
  // tile tables and item counters come from the align, which had completed
  // before the preceding launch let this one start, and the weights are
  // inputs, so the producer streams the weight blocks of its first stages
  // while the preceding kernel drains and waits before the first token rows.
  const bool early = !PAIR && p.early_weights && (warp == 0 || warp == kSchedWarp);
  if (!early) grid_dependency_wait();
  grid_dependency_trigger();
  const uint32_t tmem_base = *tmem_holder;

  const int n_tiles = p.hdr->n_tiles;
  const int n_sh = p.r > 0 ? p.hdr->n_shrink : 0;
  // CTA pairs interleave the shrink items with the first split's groups (the
  // two-phase launch runs on single-CTA tiles only)
  // (a tile's shrink slots come one wave of items before its main items:
  // `ahead` tiles of n_m weight tiles each cover the launch's work units)
  const int shs = PAIR && SPREAD && n_sh > 0 ? min(p.hdr->sh_max, n_sh) : 0;
  const int units = PAIR ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);
  const int ahead = shs > 0 ? min(n_tiles, max(1, (units + p0.n_mtiles - 1) / p0.n_mtiles)) : 0;
  const ItemOrder ord0{n_sh, n_tiles, p0.n_mtiles, shs, ahead};
  const ItemOrder ord1{n_sh, n_tiles, p1.n_mtiles, 0, 0};
  const int items0 = shs > 0 ? ahead * shs + n_tiles * (p0.n_mtiles + shs) +
                                   n_tiles * p0.n_mtiles * (p0.ksplit - 1)
                             : n_sh + n_tiles * p0.n_mtiles * p0.ksplit;
  const int n_items = items0 + (n_phases > 1 ? n_sh + n_tiles * p1.n_mtiles * p1.ksplit : 0);
  const int spc = p.r > 0 ? 128 / p.r : 0;    // shrink slots per CTA
  // shrink completions a tile's item waits for: every CTA of the item signals
  const int done_scale = PAIR ? 2 : 1;

  // Ring entries: on CTA pairs the leader writes the peer's entries too, so
  // the peer's consumers wait on "written" with a cluster-scope acquire and
  // release an entry on the leader's barrier (remotely); the leader's own
  // consumers keep CTA-scope waits and arrives, which cost less per item.
  const bool remote_ring = PAIR && !leader;
  const uint32_t iteme_rel0 = remote_ring ? mapa_shared(smem_u32(&iteme_bar[0]), 0) : 0;
  auto entry_written = [&](int q, uint32_t parity) -> bool {
    return remote_ring ? mbar_wait_cluster(smem_u32(&itemf_bar[q]), parity, abort_flag)
                       : mbar_wait(smem_u32(&itemf_bar[q]), parity, abort_flag);
  };
  auto entry_release = [&](int q) {
    if (remote_ring)
      mbar_arrive_cluster(iteme_rel0 + q * 8);
    else
      mbar_arrive(smem_u32(&iteme_bar[q]));
  };
  // Consume ring entry qc (single-thread consumers: producer, MMA issuer):
  // wait until it is written, copy it, release the slot.
  auto ring_take = [&](uint32_t qc, int& w, int& sh, TileInfo& ti, bool producer) -> bool {
    const int q = static_cast<int>(qc % kQ);
    if (!entry_written(q, (qc / kQ) & 1)) return false;
    w = ring[q].w;
    sh = ring[q].sh;
    ti = ring[q].ti;
    entry_release(q);
    if (producer && leader) mbar_arrive(smem_u32(&itemp_bar[q]));
    return true;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t cnt = 0;
      bool ok = true;
      // one TMA load of `bytes` into the current stage of this CTA's shared
      // memory, counted on the leader's full barrier when paired; the bytes
      // add up in `stage_bytes` and go to the stage's accounting once the
      // stage is issued (for an exact wind-down after an abort)
      int stage_bytes = 0;
      auto load2 = [&](uint32_t bytes, uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y) {
        stage_bytes += static_cast<int>(bytes);
        if (PAIR) tma_load_2d_pair(dst, m, fb, x, y); else tma_load_2d(dst, m, fb, x, y);
      };
      auto load3 = [&](uint32_t bytes, uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y,
                       int z) {
        stage_bytes += static_cast<int>(bytes);
        if (PAIR) tma_load_3d_pair(dst, m, fb, x, y, z); else tma_load_3d(dst, m, fb, x, y, z);
      };
      auto load4 = [&](uint32_t bytes, uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y,
                       int z, int w) {
        stage_bytes += static_cast<int>(bytes);
        if (PAIR) tma_load_4d_pair(dst, m, fb, x, y, z, w); else tma_load_4d(dst, m, fb, x, y, z, w);
      };
      auto load5 = [&](uint32_t bytes, uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y,
                       int z, int w, int v) {
        stage_bytes += static_cast<int>(bytes);
        if (PAIR) tma_load_5d_pair(dst, m, fb, x, y, z, w, v); else tma_load_5d(dst, m, fb, x, y, z, w, v);
      };
      auto stage_issued = [&](int s) {
        st_bytes[s] = stage_bytes;
        stage_bytes = 0;
      };
      // the leader's byte count of stage s for this use of it
      auto post = [&](int s, uint32_t bytes) {
        po_gen[s] = static_cast<int>(cnt);
        po_bytes[s] = static_cast<int>(bytes);
        mbar_arrive_expect_tx(smem_u32(&full_bar[s]), bytes);
      };
      // Deferred token rows.  Before the grid dependency wait (first item,
      // unpaired tiles), or before its tile's activations are complete (a
      // down item of the two-phase launch), a stage gets its weight blocks
      // and its barrier's byte count; the token rows of those stages (the
      // n_def ring slots from def_s0 on, K chunk i of the item = kc0 + i
      // rotated by rot within nkc) are loaded after the wait, which comes
      // once the ring is full or the item's K loop ends.
      bool waited = !early;
      int n_def = 0;
      int def_s0 = 0;
      const int* defer_cnt = nullptr;   // NULL: wait for the preceding launch
      int defer_target = 0;
      bool defer_ok = true;
      auto load_deferred_rows = [&](int nkc, int kc0, int rot, const CUtensorMap* tb, int brow0,
                                    int brows) -> bool {
        if (defer_cnt) {
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_gpu(defer_cnt) < defer_target) {
            if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
              defer_ok = false;
              break;
            }
            __nanosleep(64);
          }
          fence_proxy_async_global();
          defer_cnt = nullptr;
        } else {
          grid_dependency_wait();
        }
        if (defer_ok) {
          for (int d = 0; d < n_def; ++d) {
            const int s = def_s0 + d < C::kStages ? def_s0 + d : def_s0 + d - C::kStages;
            const uint32_t st = smem_u32(smem + s * C::kStageBytes);
            const uint32_t fb = smem_u32(&full_bar[s]);
            for (int j = 0; j < C::kKB && d * C::kKB + j < nkc; ++j) {
              const int i = d * C::kKB + j;
              const int kc = kc0 + (i + rot < nkc ? i + rot : i + rot - nkc);
              st_bytes[s] += brows * C::kBK * 2;   // (a stage issued earlier)
              if (PAIR) tma_load_2d_pair(st + C::b_off(j), tb, fb, kc * C::kBK, brow0);
              else tma_load_2d(st + C::b_off(j), tb, fb, kc * C::kBK, brow0);
            }
          }
        }
        waited = true;
        return defer_ok;
      };
      // stage s of this CTA is free: wait on its empty barrier; the barrier
      // that counts the stage's bytes is the leader's full barrier
      auto acquire = [&](int s, uint32_t ph, uint32_t& fb) -> bool {
        if (!mbar_try_wait(smem_u32(&empty_bar[s]), ph ^ 1) &&
            !mbar_wait(smem_u32(&empty_bar[s]), ph ^ 1, abort_flag))
          return false;
        fb = PAIR ? mapa_shared(smem_u32(&full_bar[s]), 0) : smem_u32(&full_bar[s]);
        st_gen[s] = static_cast<int>(cnt);
        return true;
      };
      // stage and phase of stage count cnt, kept running (no division)
      int sidx = 0;
      uint32_t sph = 0;
      auto advance = [&]() {
        ++cnt;
        if (++sidx == C::kStages) {
          sidx = 0;
          sph ^= 1;
        }
      };
      for (uint32_t qc = 0; ok; ++qc) {
        int w, wsh;
        TileInfo ti;
        if (!(ok = ring_take(qc, w, wsh, ti, true))) break;
        if (w < 0) break;
        const int ph = NPH == 2 && w >= items0 ? 1 : 0;
        const GemmParams& p = NPH == 2 && ph ? p1 : p0;
        const GemmMaps& maps = NPH == 2 && ph ? maps1 : maps0;
        const Item it = item_of(w - (ph ? items0 : 0), wsh, ph ? ord1 : ord0, ti.grp, p.shrink);
        const int nk = (p.K + C::kBK - 1) / C::kBK;   // K blocks of the base GEMM
        const bool gate_up = p.mode == kModeGateUp;
        if (p.act_wait) {
          // a down item of the two-phase launch: its token rows are the
          // tile's activations, complete once every gate_up item of the tile
          // has counted.  Ready: make them visible to TMA.  Not yet: stream
          // the item's weight blocks and defer its token rows to the wait.
          if (ld_acquire_gpu(&p.act_wait[it.tile]) >= p.act_target) {
            fence_proxy_async_global();
          } else {
            waited = false;
            n_def = 0;
            def_s0 = sidx;
            defer_cnt = &p.act_wait[it.tile];
            defer_target = p.act_target;
          }
        }
        const int nmma = (ti.nrows + 15) & ~15;
        const int nh = PAIR ? nmma / 2 : nmma;          // token rows this CTA loads
        const int bi = box_index(nh);
        const int brows = 16 << bi;
        const CUtensorMap* tb = &maps.b[bi];
        const int brow0 = ti.row0 + static_cast<int>(rank) * nh;
        if (it.shrink) {
          const ShrinkItem si = p.shrink[it.sh];
          // this CTA stacks slots [rank*spc, rank*spc + ns_me) of the item
          const int ns0 = min(spc, si.nslot);
          const int ns1 = PAIR ? max(0, si.nslot - spc) : 0;
          const int ns_me = rank == 0 ? ns0 : ns1;
          const uint32_t per_kb = (ns0 + ns1) * p.r * C::kBK * 2 + (PAIR ? 2 : 1) * brows * C::kBK * 2;
          // a full set of slots on consecutive adapters comes in one box of
          // 128 rows (small per-adapter boxes had made shrink items slow)
          int a_run = -1;
          if (ns_me == spc) {
            const int* sa = p.slot_adapter + si.slot0 + static_cast<int>(rank) * spc;
            a_run = sa[0];
            for (int q = 1; q < ns_me; ++q)
              if (sa[q] != a_run + q) a_run = -1;
          }
          // this item's K split of the shrink
          const int kb_lo = split_begin(nk, si.ks, p.sh_splits);
          const int kb_hi = split_begin(nk, si.ks + 1, p.sh_splits);
          for (int kb0 = kb_lo; kb0 < kb_hi && ok; kb0 += C::kKB, advance()) {
            const int nkb = min(C::kKB, kb_hi - kb0);
            const int s = sidx;
            uint32_t fb;
            if (!(ok = acquire(s, sph, fb))) break;
            const uint32_t st = smem_u32(smem + s * C::kStageBytes);
            if (leader) post(s, nkb * per_kb);
            for (int j = 0; j < nkb; ++j) {
              const int kc = kb0 + j;
              if (a_run >= 0) {
                load4(spc * p.r * C::kBK * 2, st + C::a_off(j), &maps.la_run, fb, kc * C::kBK, 0, ti.expert,
                      a_run);
              } else {
                for (int q = 0; q < ns_me; ++q)
                  load4(p.r * C::kBK * 2, st + C::a_off(j) + q * p.r * C::kBK * 2, &maps.la, fb, kc * C::kBK,
                        0, ti.expert, p.slot_adapter[si.slot0 + static_cast<int>(rank) * spc + q]);
              }
              if (waited) load2(brows * C::kBK * 2, st + C::b_off(j), tb, fb, kc * C::kBK, brow0);
            }
            stage_issued(s);
            if (!waited && ++n_def == C::kStages && !load_deferred_rows(kb_hi - kb_lo, kb_lo, 0, tb, brow0, brows))
              ok = false;
          }
          if (ok && !waited && !load_deferred_rows(kb_hi - kb_lo, kb_lo, 0, tb, brow0, brows)) ok = false;
        } else {
          const uint32_t per_kb = (PAIR ? 2 : 1) * (C::kATile + brows * C::kBK * 2);
          const int kc0 = p.split_k0[it.ks];
          const int nkc = p.split_k0[it.ks + 1] - kc0;
          // (paired tiles, tensor-bound: the token tiles of one expert read
          // the same weight blocks at the same time, so no rotation there)
          const int rot = PAIR ? 0 : k_rotation(it, nkc);
          // this CTA's 128 weight rows: gate_up features m*64*(1+PAIR) + rank*64,
          // down / linear rows m*kMRows + rank*128
          const int grow = gate_up ? it.m * (PAIR ? 128 : 64) + static_cast<int>(rank) * 64
                                   : it.m * C::kMRows + static_cast<int>(rank) * 128;
          for (int i0 = 0; i0 < nkc && ok; i0 += C::kKB, advance()) {
            const int nkb = min(C::kKB, nkc - i0);
            const int s = sidx;
            uint32_t fb;
            if (!(ok = acquire(s, sph, fb))) break;
            const uint32_t st = smem_u32(smem + s * C::kStageBytes);
            if (leader) post(s, nkb * per_kb);
            for (int j = 0; j < nkb; ++j) {
              const int i = i0 + j;
              const int kc = kc0 + (i + rot < nkc ? i + rot : i + rot - nkc);
              if (gate_up)   // 64 features, each gate row followed by its up row, in one box
                load4(C::kATile, st + C::a_off(j), &maps.w, fb, kc * C::kBK, 0, grow, ti.expert);
              else
                load3(C::kATile, st + C::a_off(j), &maps.w, fb, kc * C::kBK, grow, ti.expert);
              if (waited) load2(brows * C::kBK * 2, st + C::b_off(j), tb, fb, kc * C::kBK, brow0);
            }
            stage_issued(s);
            if (!waited && ++n_def == C::kStages && !load_deferred_rows(nkc, kc0, rot, tb, brow0, brows))
              ok = false;
          }
          if (ok && !waited && !load_deferred_rows(nkc, kc0, rot, tb, brow0, brows)) ok = false;
          if (ok && p.r > 0 && ti.nslots > 0 && it.ks == p.ksplit - 1) {
            // the tile's shrink results must be complete and visible to TMA
            const int target = p.done_target * ti.nsh * done_scale;
            const uint64_t t0 = globaltimer_ns();
            while (ld_acquire_gpu(&p.tile_done[it.tile]) < target) {
              if (*abort_flag || globaltimer_ns() - t0 > kWaitLimitNs) {
                ok = false;
                break;
              }
              __nanosleep(64);
            }
            fence_proxy_async_global();
            const CUtensorMap* tz = &maps.z[bi];
            const int lw = p.lora_w;
            // expand chunks: (slot, chunk, part), the part (hi, lo) fastest so
            // that a LoRA B chunk is read twice in a row (the second from L2)
            const int nl = ti.nslots * p.lora_chunks * p.z_parts;
            const uint32_t per_sub = (PAIR ? 2 : 1) * (128 * lw * 2 + brows * lw * 2);
            const int cps = C::kKB * C::kBK / lw;       // chunks packed per stage
            for (int i0 = 0; i0 < nl && ok; i0 += cps, advance()) {
              const int nsub = min(cps, nl - i0);
              const int s = sidx;
              uint32_t fb;
              if (!(ok = acquire(s, sph, fb))) break;
              const uint32_t st = smem_u32(smem + s * C::kStageBytes);
              if (leader) post(s, nsub * per_sub);
              for (int j = 0; j < nsub; ++j) {
                const int per_slot = p.lora_chunks * p.z_parts;
                const int sl = (i0 + j) / per_slot;
                const int cp = (i0 + j) - sl * per_slot;
                const int c = cp / p.z_parts;
                const int part = cp - c * p.z_parts;
                // (a failed check loads slot 0's data instead: the stage still
                // receives the bytes its barrier expects)
                const int sidx_ok =
                    MOELORA_IN_RANGE(p.err, ti.slot_base + sl, 0, p.zpart_slots) ? ti.slot_base + sl : 0;
                const int a = p.slot_adapter[sidx_ok];
                if (gate_up)
                  load5(128 * lw * 2, st + C::lora_a_off(j, lw), &maps.lb, fb, c * lw, 0, grow, ti.expert,
                        a);
                else
                  load4(128 * lw * 2, st + C::lora_a_off(j, lw), &maps.lb, fb, c * lw, grow, ti.expert, a);
                load2(brows * lw * 2, st + C::lora_b_off(j, lw), tz, fb, part * p.r + c * lw,
                      (ti.slot_base + sl) * TN + static_cast<int>(rank) * nh);
              }
              stage_issued(s);
            }
          }
        }
      }
      if (!ok) {
        // (the copies already issued are waited for at the end of the kernel)
        *abort_flag = 1;
        flag_error(p.err, kStatusTimeout);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      int sidx = 0;            // stage of the next MMA batch, and its full-barrier phase
      uint32_t sph = 0;
      const uint32_t smem0 = smem_u32(smem);
      uint32_t li = 0;
      bool ok = true;
      bool issued = false;
      for (uint32_t qc = 0; ok; ++qc, ++li) {
        int w, wsh;
        TileInfo ti;
        if (!(ok = ring_take(qc, w, wsh, ti, false))) break;
        if (w < 0) break;
        const int ph = NPH == 2 && w >= items0 ? 1 : 0;
        const GemmParams& p = NPH == 2 && ph ? p1 : p0;
        const Item it = item_of(w - (ph ? items0 : 0), wsh, ph ? ord1 : ord0, ti.grp, p.shrink);
        const int nk = (p.K + C::kBK - 1) / C::kBK;
        const int nmma = (ti.nrows + 15) & ~15;
        const uint32_t idesc = make_idesc_bf16(nmma, PAIR ? 256 : 128);
        const int buf = li & 1;
        if (!(ok = mbar_wait(smem_u32(&acce_bar[buf]), ((li >> 1) & 1) ^ 1, abort_flag))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * TN;
        const int nl =
            (!it.shrink && p.r > 0 && it.ks == p.ksplit - 1) ? ti.nslots * p.lora_chunks * p.z_parts : 0;
        int nb;
        if (it.shrink) {
          const int sks = p.shrink[it.sh].ks;
          nb = split_begin(nk, sks + 1, p.sh_splits) - split_begin(nk, sks, p.sh_splits);
        } else {
          nb = p.split_k0[it.ks + 1] - p.split_k0[it.ks];
        }
        const int st_base = (nb + C::kKB - 1) / C::kKB;
        const int cps = p.r > 0 ? C::kKB * C::kBK / p.lora_w : 1;   // expand chunks per stage
        const int st_all = st_base + (nl + cps - 1) / cps;
        uint32_t acc = 0;   // the item's first MMA overwrites the accumulator
        // The issuing thread blocks on each MMA (the queue holds about one),
        // so the work between two MMAs is kept small: descriptors of a stage
        // are a base plus constant offsets (the 14-bit start field of a
        // descriptor is the byte address / 16, and every operand of the
        // shared-memory window stays inside it), and full base stages run
        // an unrolled loop.
        for (int sti = 0; sti < st_all; ++sti) {
          const int s = sidx;
          const uint32_t ph = sph;
          if (!mbar_try_wait(smem_u32(&full_bar[s]), ph) &&
              !(ok = mbar_wait(smem_u32(&full_bar[s]), ph, abort_flag)))
            break;
          tc_fence_after();
          const uint32_t st = smem0 + s * C::kStageBytes;
          if (sti < st_base) {   // base GEMM: K blocks of kBK (kBK / 16 MMAs of K=16 each)
            const uint64_t ad0 = make_smem_desc(st + C::a_off(0), C::kSboK, C::kSwzK);
            const uint64_t bd0 = make_smem_desc(st + C::b_off(0), C::kSboK, C::kSwzK);
            const int nsub = min(C::kKB, nb - sti * C::kKB);
            if (nsub == C::kKB) {
#pragma unroll
              for (int j = 0; j < C::kKB; ++j) {
#pragma unroll
                for (int kk = 0; kk < C::kBK / 16; ++kk) {
                  const uint64_t ad = ad0 + static_cast<uint64_t>((C::a_off(j) + kk * 32) >> 4);
                  const uint64_t bd = bd0 + static_cast<uint64_t>((j * C::kBTileBytes + kk * 32) >> 4);
                  if (PAIR) mma_bf16_pair(d_tmem, ad, bd, idesc, acc); else mma_bf16(d_tmem, ad, bd, idesc, acc);
                  acc = 1;
                }
              }
            } else {
              for (int j = 0; j < nsub; ++j) {
#pragma unroll
                for (int kk = 0; kk < C::kBK / 16; ++kk) {
                  const uint64_t ad = ad0 + static_cast<uint64_t>((C::a_off(j) + kk * 32) >> 4);
                  const uint64_t bd = bd0 + static_cast<uint64_t>((j * C::kBTileBytes + kk * 32) >> 4);
                  if (PAIR) mma_bf16_pair(d_tmem, ad, bd, idesc, acc); else mma_bf16(d_tmem, ad, bd, idesc, acc);
                  acc = 1;
                }
              }
            }
          } else {   // LoRA expand: chunks of width lora_w packed by bytes
            const int lw = p.lora_w;
            const uint32_t swz = static_cast<uint32_t>(p.lora_swz);
            const uint32_t sbo = static_cast<uint32_t>(8 * lw * 2);
            const int nsub = min(cps, nl - (sti - st_base) * cps);
            const uint64_t ad0 = make_smem_desc(st + C::lora_a_off(0, lw), sbo, swz);
            const uint64_t bd0 = make_smem_desc(st + C::lora_b_off(0, lw), sbo, swz);
            for (int j = 0; j < nsub; ++j) {
              for (int kk = 0; kk < lw / 16; ++kk) {
                const uint64_t ad = ad0 + static_cast<uint64_t>((C::lora_a_off(j, lw) + kk * 32) >> 4);
                const uint64_t bd =
                    bd0 + static_cast<uint64_t>((C::lora_b_off(j, lw) - C::lora_b_off(0, lw) + kk * 32) >> 4);
                if (PAIR) mma_bf16_pair(d_tmem, ad, bd, idesc, acc); else mma_bf16(d_tmem, ad, bd, idesc, acc);
                acc = 1;
              }
            }
          }
          issued = true;
          if (PAIR) mma_commit_pair(smem_u32(&empty_bar[s])); else mma_commit(smem_u32(&empty_bar[s]));
          if (++sidx == C::kStages) {
            sidx = 0;
            sph ^= 1;
          }
        }
        if (ok) {
          if (PAIR) mma_commit_pair(smem_u32(&accf_bar[buf])); else mma_commit(smem_u32(&accf_bar[buf]));
        }
      }
      if (!ok) {
        *abort_flag = 1;
        flag_error(p.err, kStatusTimeout);
      }
      if (!ok && issued) {
        // wait (bounded) for the MMAs in flight before TMEM is released
        if (PAIR) mma_commit_pair(smem_u32(drain_bar)); else mma_commit(smem_u32(drain_bar));
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(drain_bar), 0))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------ item scheduler
    // Writes the CTA's item sequence into the ring, claiming items from the
    // launch's counter as it goes: items cost about the same, but SMs stream
    // from HBM at different rates, and a fixed share leaves the slowest SMs
    // the tail (decode 0.266 -> 0.261 ms, dense T=1 0.103 -> 0.094 ms on
    // GB300).  On CTA pairs the leader claims for the pair and writes the
    // peer's ring entry as well (the peer's scheduler has nothing to do).
    // Items are claimed in index order by CTAs that are running, and a
    // tile's shrink items precede its main items in either order, so they
    // are always claimed, and finished, by resident CTAs before any main item
    // that waits for them: no wait depends on a CTA (pair) that has not
    // started, however many of the grid's CTAs are resident.
    if (lane == 0 && leader) {
      bool ok = true;
      const uint32_t peer_ring = PAIR ? mapa_shared(smem_u32(ring), 1) : 0;
      const uint32_t peer_itemf = PAIR ? mapa_shared(smem_u32(&itemf_bar[0]), 1) : 0;
      for (uint32_t qp = 0;; ++qp) {
        const int q = static_cast<int>(qp % kQ);
        // every consumer (of both CTAs) has read the entry's previous use
        if (!(ok = PAIR ? mbar_wait_cluster(smem_u32(&iteme_bar[q]), ((qp / kQ) & 1) ^ 1, abort_flag)
                        : mbar_wait(smem_u32(&iteme_bar[q]), ((qp / kQ) & 1) ^ 1, abort_flag)))
          break;
        // claim no further ahead than kClaimAhead items past the producer, so
        // that the items left go to whichever CTA runs out first
        if (qp >= static_cast<uint32_t>(kClaimAhead)) {
          const uint32_t e = qp - kClaimAhead;
          if (!(ok = mbar_wait(smem_u32(&itemp_bar[e % kQ]), (e / kQ) & 1, abort_flag))) break;
        }
        int w, wsh = -1;
        TileInfo ti = {};
        for (;;) {
          w = atomicAdd(p.work_ctr, 1);
          if (w >= n_items) {
            w = -1;
            break;
          }
          const bool w1 = NPH == 2 && w >= items0;
          const GemmParams& pw = w1 ? p1 : p0;
          int tile;
          // (an empty shrink slot of the spread order: claim the next item)
          if (resolve_item(w - (w1 ? items0 : 0), w1 ? ord1 : ord0, p.tiles, p.shrink, pw.sh_splits, wsh,
                           tile)) {
            ti = p.tiles[tile];
            break;
          }
        }
        ring[q].ti = ti;
        ring[q].w = w;
        ring[q].sh = wsh;
        if (PAIR) {
          // the peer's copy of the entry, released by its "written" arrive
          const uint32_t dst = peer_ring + q * static_cast<uint32_t>(sizeof(RingEntry));
          st_cluster_u32(dst, static_cast<uint32_t>(w));
          if (shs > 0)   // (all shrink entries first: the peer decodes them from w)
            st_cluster_u32(dst + static_cast<uint32_t>(offsetof(RingEntry, sh)), static_cast<uint32_t>(wsh));
          const uint32_t* tv = reinterpret_cast<const uint32_t*>(&ti);
#pragma unroll
          for (int i = 0; i < static_cast<int>(sizeof(TileInfo) / 4); ++i)
            st_cluster_u32(dst + static_cast<uint32_t>(offsetof(RingEntry, ti)) + 4 * i, tv[i]);
          mbar_arrive_cluster(peer_itemf + q * 8);
        }
        mbar_arrive(smem_u32(&itemf_bar[q]));
        if (w < 0) break;
      }
      if (!ok) {
        *abort_flag = 1;
        flag_error(p.err, kStatusTimeout);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;     // accumulator row = weight row of this CTA's half
    // the MMA issuer's "accumulator free" barrier (the leader's, when paired)
    const uint32_t acce0 = PAIR ? mapa_shared(smem_u32(&acce_bar[0]), 0) : smem_u32(&acce_bar[0]);
    uint32_t li = 0;
    for (uint32_t qc = 0;; ++qc, ++li) {
      // the next ring entry: every epilogue thread reads it, the warps agree
      // on the outcome of the wait, and each warp releases the slot
      const int q = static_cast<int>(qc % kQ);
      const bool got = entry_written(q, (qc / kQ) & 1);
      if (bar_red_or(1, 128, !got || *abort_flag)) {
        if (!got) flag_error(p.err, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      const int w = ring[q].w;
      const int wsh = ring[q].sh;
      const TileInfo ti = ring[q].ti;
      __syncwarp();
      if (lane == 0) entry_release(q);
      if (w < 0) break;
      const int ph = NPH == 2 && w >= items0 ? 1 : 0;
      const GemmParams& p = NPH == 2 && ph ? p1 : p0;
      const Item it = item_of(w - (ph ? items0 : 0), wsh, ph ? ord1 : ord0, ti.grp, p.shrink);
      const bool gate_up = p.mode == kModeGateUp;
      const int nmma = (ti.nrows + 15) & ~15;
      const int buf = li & 1;
      const bool ok = mbar_wait(smem_u32(&accf_bar[buf]), (li >> 1) & 1, abort_flag);
      if (bar_red_or(1, 128, !ok || *abort_flag)) {
        if (!ok) flag_error(p.err, kStatusTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t t_row = tmem_base + buf * TN + (static_cast<uint32_t>(quarter * 32) << 16);

      if (it.shrink) {
        const ShrinkItem si = p.shrink[it.sh];
        const int j = static_cast<int>(rank) * spc + row / p.r;   // slot of the item
        const int q = row % p.r;
        const bool valid = j < si.nslot && row / p.r < spc &&
                           MOELORA_IN_RANGE(p.err, si.slot0 + j, 0, p.zpart_slots) &&
                           MOELORA_IN_RANGE(p.err, ti.expert, 0, p.n_experts);
        const int a_j = valid ? p.slot_adapter[si.slot0 + j] : -3;
        __nv_bfloat16* zrow =
            p.zbuf + (static_cast<size_t>(si.slot0 + (valid ? j : 0)) * TN) * (p.z_parts * p.r) + q;
        // the slot's tokens: rows of one expert are sorted by adapter, so they
        // are the tile's columns [c_lo, c_hi) of the (expert, adapter) bin
        int c_lo = 0, c_hi = 0;
        if (valid) {
          const int b = ti.expert * p.lp1 + a_j + 1;
          c_lo = p.bin_start[b] - ti.row0;
          c_hi = a_j + 2 < p.lp1 ? p.bin_start[b + 1] - ti.row0 : ti.nrows;
          c_hi = min(c_hi, ti.nrows);
        }
        // z of columns c0 .. c0+15 (the slot's tokens kept, zeros elsewhere)
        auto store_z = [&](const float* v, int c0) {
#pragma unroll
          for (int cc = 0; cc < 16; ++cc) {
            const int c = c0 + cc;
            const bool keep = c >= c_lo && c < c_hi;
            const float z = keep ? v[cc] : 0.0f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(z);
            zrow[static_cast<size_t>(c) * (p.z_parts * p.r)] = hi;
            if (p.z_parts == 2)
              zrow[static_cast<size_t>(c) * (2 * p.r) + p.r] = __float2bfloat16_rn(z - __bfloat162float(hi));
          }
        };
        bool last = true;
        if (p.sh_splits == 1) {
          for (int c0 = 0; c0 < nmma; c0 += 16) {
            float v[16];
            tmem_ld16(t_row + c0, v);
            if (valid) store_z(v, c0);
          }
        } else {
          // K split: this split's fp32 part of every column, then its
          // arrival; the split that arrives last (whichever it is) sums the
          // parts in split order, so the result does not depend on timing
          const size_t slot = static_cast<size_t>(si.slot0 + (valid ? j : 0));
          float* part = p.zpart + ((static_cast<size_t>(si.ks) * p.zpart_slots + slot) * TN) * p.r + q;
          for (int c0 = 0; c0 < nmma; c0 += 16) {
            float v[16];
            tmem_ld16(t_row + c0, v);
            if (valid) {
#pragma unroll
              for (int cc = 0; cc < 16; ++cc) part[static_cast<size_t>(c0 + cc) * p.r] = v[cc];
            }
          }
          named_bar_sync(1, 128);
          bool mine = false;
          if (row == 0) {
            __threadfence();
            const int before =
                atomicAdd(&p.sh_cnt[2 * (it.sh / p.sh_splits) + static_cast<int>(rank)], 1);
            mine = before + 1 == p.done_target * p.sh_splits;
            __threadfence();
          }
          last = bar_red_or(1, 128, mine);
          if (last && valid) {
            for (int c0 = 0; c0 < nmma; c0 += 16) {
              float v[16];
#pragma unroll
              for (int cc = 0; cc < 16; ++cc) v[cc] = 0.0f;
              for (int s = 0; s < p.sh_splits; ++s) {
                const float* ps = p.zpart + ((static_cast<size_t>(s) * p.zpart_slots + slot) * TN) * p.r + q;
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) v[cc] += __ldcg(ps + static_cast<size_t>(c0 + cc) * p.r);
              }
              store_z(v, c0);
            }
          }
        }
        if (last) {
          // publish: every epilogue thread's stores, then one release
          named_bar_sync(1, 128);
          if (row == 0) {
            __threadfence();
            fence_proxy_async_global();
            atomicAdd(&p.tile_done[it.tile], 1);
          }
        }
      } else if (gate_up) {
        // TMEM lane 2i holds gate row i and lane 2i+1 the up row of the same
        // feature (the weight box interleaves them), so a feature's two
        // accumulator rows sit in adjacent threads of one warp.  Per chunk of
        // W columns the gate thread finishes the first W/2 columns and the up
        // thread the last W/2, each taking the values it lacks from its
        // partner by one lane shuffle.
        const bool is_gate = (row & 1) == 0;
        const int feat = it.m * (PAIR ? 128 : 64) + static_cast<int>(rank) * 64 + (row >> 1);
        __nv_bfloat16* orow = p.out + static_cast<size_t>(ti.row0) * p.out_ld + feat;
        const bool store_ok = feat < p.out_feats;
        auto finish = [&](const float* v, int c0, int half) {
          // v: this thread's W = 2*half values of columns c0 .. c0+W-1
          const int cbase = c0 + (is_gate ? 0 : half);
#pragma unroll
          for (int cc = 0; cc < half; ++cc) {
            // the gate thread hands over its gate values of the up thread's
            // columns, the up thread its up values of the gate thread's
            const float other = __shfl_xor_sync(0xffffffffu, is_gate ? v[half + cc] : v[cc], 1);
            const float g = is_gate ? v[cc] : other;
            const float u = is_gate ? other : v[half + cc];
            const int c = cbase + cc;
            if (store_ok && c < ti.nrows && MOELORA_IN_RANGE(p.err, ti.row0 + c, 0, p.Pmax))
              orow[static_cast<size_t>(c) * p.out_ld] = __float2bfloat16_rn(silu_f(g) * u);
          }
        };
        bool last = true;
        if (p.ksplit > 1) {
          // K split: this split's fp32 part of every column, then its
          // arrival; the split that arrives last (whichever it is) sums the
          // parts in split order, so the result does not depend on timing
          const size_t slot = static_cast<size_t>(it.tile) * p.n_mtiles + it.m;
          auto part_of = [&](int s) {
            return p.gu_part + ((static_cast<size_t>(s) * p.gu_slots + slot) * 128 + row) * TN;
          };
          float* mine_part = part_of(it.ks);
          for (int c0 = 0; c0 < nmma; c0 += 16) {
            float v[16];
            tmem_ld16(t_row + c0, v);
#pragma unroll
            for (int cc = 0; cc < 16; cc += 4)
              *reinterpret_cast<float4*>(mine_part + c0 + cc) = make_float4(v[cc], v[cc + 1], v[cc + 2], v[cc + 3]);
          }
          named_bar_sync(1, 128);
          bool mine = false;
          if (row == 0) {
            __threadfence();
            mine = atomicAdd(&p.gu_cnt[slot], 1) + 1 == p.ksplit;
            __threadfence();
          }
          last = bar_red_or(1, 128, mine);
          if (last) {
            int c0 = 0;
            for (; c0 + 32 <= nmma; c0 += 32) {
              float v[32];
#pragma unroll
              for (int cc = 0; cc < 32; ++cc) v[cc] = 0.0f;
              for (int s = 0; s < p.ksplit; ++s) {
                const float4* ps = reinterpret_cast<const float4*>(part_of(s) + c0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  const float4 w = __ldcg(ps + q);
                  v[4 * q] += w.x;
                  v[4 * q + 1] += w.y;
                  v[4 * q + 2] += w.z;
                  v[4 * q + 3] += w.w;
                }
              }
              finish(v, c0, 16);
            }
            if (c0 < nmma) {   // a last chunk of 16 columns
              float v[16];
#pragma unroll
              for (int cc = 0; cc < 16; ++cc) v[cc] = 0.0f;
              for (int s = 0; s < p.ksplit; ++s) {
                const float4* ps = reinterpret_cast<const float4*>(part_of(s) + c0);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  const float4 w = __ldcg(ps + q);
                  v[4 * q] += w.x;
                  v[4 * q + 1] += w.y;
                  v[4 * q + 2] += w.z;
                  v[4 * q + 3] += w.w;
                }
              }
              finish(v, c0, 8);
            }
          }
        } else {
          int c0 = 0;
          for (; c0 + 32 <= nmma; c0 += 32) {
            float v[32];
            tmem_ld32(t_row + c0, v);
            finish(v, c0, 16);
          }
          if (c0 < nmma) {   // a last chunk of 16 columns
            float v[16];
            tmem_ld16(t_row + c0, v);
            finish(v, c0, 8);
          }
        }
        if (last && p.act_count) {
          // two-phase launch: publish this item's activation rows to the
          // tile's down items (every thread's stores, then one release)
          named_bar_sync(1, 128);
          if (row == 0) {
            __threadfence();
            fence_proxy_async_global();
            atomicAdd(&p.act_count[it.tile], 1);
          }
        }
      } else {
        const int feat = it.m * C::kMRows + static_cast<int>(rank) * 128 + row;
        const bool linear = p.mode == kModeLinear;
        for (int c0 = 0; c0 < nmma; c0 += 16) {
          float v[16];
          tmem_ld16(t_row + c0, v);
          if (feat < p.out_feats) {
#pragma unroll
            for (int cc = 0; cc < 16; ++cc) {
              const int c = c0 + cc;
              if (c < ti.nrows) {
                const int prow = ti.row0 + c;
                if (!MOELORA_IN_RANGE(p.err, prow, 0, p.Pmax)) continue;
                if (linear) {
                  const int t = p.row_tok[prow];
                  if (MOELORA_IN_RANGE(p.err, t, 0, p.T))
                    p.out[static_cast<size_t>(t) * p.out_ld + feat] = __float2bfloat16_rn(v[cc]);
                } else {
                  p.out_f32[it.ks * p.split_stride + static_cast<size_t>(prow) * p.out_ld + feat] =
                      v[cc] * p.row_w[prow];
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR)
          mbar_arrive_cluster(acce0 + buf * 8);
        else
          mbar_arrive(acce0 + buf * 8);
      }
    }
  }

  __syncthreads();
  // (each CTA of a pair hands its abort flag to the other, so that both take
  // the same decision below)
  if (PAIR && threadIdx.x == 0)
    st_cluster_u32(mapa_shared(smem_u32(peer_abort), rank ^ 1), static_cast<uint32_t>(*abort_flag));
  if (PAIR) cluster_sync();   // no CTA leaves while its peer may still touch it
  const bool any_abort = *abort_flag || (PAIR && *reinterpret_cast<volatile int*>(peer_abort));
  // After an abort some copies may still be in flight into a stage whose
  // MMAs never ran.  Every producer has stopped issuing by now, and its
  // accounting says, per stage slot, what it last posted and issued: the CTA
  // that counts a slot's bytes (the leader; each CTA when unpaired) settles
  // the slot's latest phase -- posts the bytes nobody announced, or marks as
  // arrived the announced bytes nobody sent -- and waits (bounded) until the
  // copies actually issued have landed.  Nothing then writes into a CTA's
  // shared memory or barriers after it exits.
  if (warp == 0 && lane == 0 && leader) {
    if (any_abort) {
      for (int s = 0; s < C::kStages; ++s) {
        const int g_me = st_gen[s];
        const int b_me = st_bytes[s];
        const int g_pe = PAIR ? static_cast<int>(ld_cluster_u32(mapa_shared(smem_u32(&st_gen[s]), 1))) : -1;
        const int b_pe = PAIR ? static_cast<int>(ld_cluster_u32(mapa_shared(smem_u32(&st_bytes[s]), 1))) : 0;
        const int g = max(max(g_me, g_pe), po_gen[s]);
        if (g < 0) continue;
        const int arrived = (g_me == g ? b_me : 0) + (g_pe == g ? b_pe : 0);
        const uint32_t fb = smem_u32(&full_bar[s]);
        if (po_gen[s] == g) {
          if (po_bytes[s] > arrived) mbar_complete_tx(fb, static_cast<uint32_t>(po_bytes[s] - arrived));
        } else {
          mbar_arrive_expect_tx(fb, static_cast<uint32_t>(arrived));
        }
        const uint32_t parity = (static_cast<uint32_t>(g) / C::kStages) & 1;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(fb, parity))
          if (globaltimer_ns() - t0 > kWaitLimitNs) break;
      }
    }
  }
  if (PAIR && any_abort) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR)
      tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else
      tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// One phase per launch: the parameters by value, read at fixed offsets.
// SPREAD: the shrink entries spread over the first K split (CTA pairs; a
// separate instance, so that the all-first order keeps its own code).
template <int TN, bool PAIR, bool SPREAD>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmParams p) {
  gemm_body<TN, PAIR, 1, SPREAD>(maps, maps, p, p);
}

// Both phases in one launch (single-CTA tiles): the items pick their phase's
// maps and parameters, so these are grid constants (addressable in place).
template <int TN>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gemm_two_phase_kernel(const __grid_constant__ GemmMaps maps0,
                              const __grid_constant__ GemmMaps maps1,
                              const __grid_constant__ GemmParams p0,
                              const __grid_constant__ GemmParams p1) {
  gemm_body<TN, false, 2, false>(maps0, maps1, p0, p1);
}

template <int TN, bool PAIR, int NPH, bool SPREAD>
struct KernelOf {
  static constexpr auto fn = moe_gemm_kernel<TN, PAIR, SPREAD>;
};
template <int TN>
struct KernelOf<TN, false, 2, false> {
  static constexpr auto fn = moe_gemm_two_phase_kernel<TN>;
};

template <int TN, bool PAIR, int NPH, bool SPREAD = false>
cudaError_t launch_tn(const GemmMaps& maps0, const GemmParams& p0, const GemmMaps& maps1,
                      const GemmParams& p1, int grid, cudaStream_t stream) {
  using C = Cfg<TN, PAIR>;
  static_assert(C::kSmemBytes <= 232448, "shared memory budget");
  static int configured_device = -1;
  static int max_units = 0;   // co-resident CTAs (pairs count as one unit)
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(KernelOf<TN, PAIR, NPH, SPREAD>::fn,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = C::kSmemBytes;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int clusters = 0;
      e = cudaOccupancyMaxActiveClusters(&clusters, KernelOf<TN, PAIR, NPH, SPREAD>::fn, &cfg);
      if (e != cudaSuccess) return e;
      max_units = clusters;
    } else {
      int per_sm = 0, sms = 0;
      e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, KernelOf<TN, PAIR, NPH, SPREAD>::fn, kThreads,
                                                        C::kSmemBytes);
      if (e != cudaSuccess) return e;
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      max_units = per_sm * sms;
    }
    if (max_units < 1) return cudaErrorInvalidConfiguration;
    configured_device = dev;
  }
  // no more CTAs (pairs) than fit at once: a persistent CTA beyond that
  // would only start when another ends
  const int units = std::max(1, std::min(grid, max_units));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PAIR ? 2 * units : units);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int na = 1;
  if (PAIR) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    na = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  if constexpr (NPH == 2)
    return cudaLaunchKernelEx(&cfg, KernelOf<TN, PAIR, NPH, SPREAD>::fn, maps0, maps1, p0, p1);
  else
    return cudaLaunchKernelEx(&cfg, KernelOf<TN, PAIR, NPH, SPREAD>::fn, maps0, p0);
}

}  // namespace

size_t moe_gemm_smem_bytes(int tn) {
  return tn >= 256 ? Cfg<256, true>::kSmemBytes
                   : (tn >= 128 ? Cfg<128, false>::kSmemBytes
                                : (tn >= 64 ? Cfg<64, false>::kSmemBytes
                                            : (tn >= 32 ? Cfg<32, false>::kSmemBytes
                                                        : Cfg<16, false>::kSmemBytes)));
}

bool moe_gemm_paired(int tn) { return tn >= 256; }

int moe_gemm_kblock_width(int tn) {
  return tn >= 256 ? Cfg<256, true>::kBK : Cfg<16, false>::kBK;
}

int moe_gemm_stage_kblocks(int tn) {
  return tn >= 256 ? Cfg<256, true>::kKB
                   : (tn >= 128 ? Cfg<128, false>::kKB
                                : (tn >= 64 ? Cfg<64, false>::kKB
                                            : (tn >= 32 ? Cfg<32, false>::kKB : Cfg<16, false>::kKB)));
}

cudaError_t launch_moe_gemm(int tn, const GemmMaps& maps, const GemmParams& p, int grid,
                            cudaStream_t stream) {
  if (tn == 256)
    return p.spread_shrink ? launch_tn<256, true, 1, true>(maps, p, maps, p, grid, stream)
                           : launch_tn<256, true, 1, false>(maps, p, maps, p, grid, stream);
  if (tn == 128) return launch_tn<128, false, 1>(maps, p, maps, p, grid, stream);
  if (tn == 64) return launch_tn<64, false, 1>(maps, p, maps, p, grid, stream);
  if (tn == 32) return launch_tn<32, false, 1>(maps, p, maps, p, grid, stream);
  if (tn == 16) return launch_tn<16, false, 1>(maps, p, maps, p, grid, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_moe_gemm_two_phase(int tn, const GemmMaps& maps0, const GemmParams& p0,
                                      const GemmMaps& maps1, const GemmParams& p1, int grid,
                                      cudaStream_t stream) {
  if (tn == 128) return launch_tn<128, false, 2>(maps0, p0, maps1, p1, grid, stream);
  if (tn == 64) return launch_tn<64, false, 2>(maps0, p0, maps1, p1, grid, stream);
  if (tn == 32) return launch_tn<32, false, 2>(maps0, p0, maps1, p1, grid, stream);
  if (tn == 16) return launch_tn<16, false, 2>(maps0, p0, maps1, p1, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace moelora
