// C ABI of the MoE-LoRA expert layer: argument checks, the workspace plan,
// TMA tensor maps and the launch sequence
//   align (hist, scan, scatter) -> permute -> gate_up GEMM phase (with its
//   LoRA shrink items) -> down GEMM phase (with its shrink items) -> combine
// all on the caller's stream, with no allocation and no synchronisation.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <fstream>
#include <sstream>
#include <string>
#include <vector>

#include <dirent.h>
#include <sys/stat.h>

#include "align.cuh"
#include "gemm_tc.cuh"
#include "merge.cuh"

using namespace moelora;

namespace {

constexpr int kBlockM = 16;          // forward: per-expert row padding = MMA N granularity
constexpr size_t kWsAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------ plan
struct Plan {
  bool linear = false;
  int T = 0, k = 0, E = 0, H = 0, I = 0, L = 0, r = 0, N = 0;  // linear: H = K, N = out
  bool lora = false;
  int n = 0, nbins = 0, nchunks = 0, block_m = kBlockM, Pmax = 0, tn = 32;
  int n_tiles_max = 0, n_slots_max = 0, n_sh_max = 0;
  int sks = 1;                        // K splits of every shrink item
  int ksplit = 1;                     // K splits of the down / linear phase
  int gksplit = 1;                    // K splits of the gate_up phase (single-CTA tiles)
  size_t off_hdr = 0, off_chunk_hist = 0, off_bin_of = 0, off_rank_of = 0, off_bin_start = 0;
  size_t off_row_tok = 0, off_row_w = 0, off_pos_of = 0;
  size_t off_tiles = 0, off_shrink = 0, off_slot_ad = 0, off_tile_done = 0;
  size_t off_sh_cnt = 0, off_zpart = 0, off_act_done = 0;
  size_t off_xperm = 0, off_zgu = 0, off_zd = 0, off_act = 0, off_ypair = 0;
  size_t off_topk_ids = 0, off_topk_w = 0;   // router results (routed forward)
  size_t off_gupart = 0, off_gucnt = 0;      // K-split gate_up parts and arrival counters
  size_t total = 0;
};

struct Bump {
  size_t cur = 0;
  size_t take(size_t bytes) {
    const size_t at = cur;
    cur = align_up(cur + bytes, kWsAlign);
    return at;
  }
};

// Tuning overrides for benchmarking: MOELORA_KSPLIT (1..4), MOELORA_TN
// (16, 32, 64, 128, 256), MOELORA_GROUP_TILES (at most this many token tiles
// per L2 group of the GEMM item order), MOELORA_GU_KSPLIT, MOELORA_TWO_PHASE,
// MOELORA_SHRINK_SPLITS, MOELORA_SPREAD_SHRINK (0 / 1) and MOELORA_PF_MB /
// MOELORA_PF_CTAS (the small align's weight prefetch).  Read at planning
// time, so the workspace size and the call agree; unset means the built-in
// choice.
int env_override(const char* name, int lo, int hi) {
  const char* v = std::getenv(name);
  if (!v) return 0;
  const int x = std::atoi(v);
  return (x >= lo && x <= hi) ? x : 0;
}

// Failure-detection test hook: with MOELORA_FAULT_INJECT=shrink_wait the
// first GEMM phase of a call (gate_up, or the dense linear's only phase)
// waits for twice the shrink completions its tiles will ever see.  Its
// bounded counter wait then runs out (after the library's 2 s wait limit),
// the kernel winds down, and moelora_get_error reports MOELORA_ERR_TIMEOUT;
// nothing faults or hangs, and the next call runs normally.
int first_phase_done_target() {
  const char* v = std::getenv("MOELORA_FAULT_INJECT");
  return v && std::strcmp(v, "shrink_wait") == 0 ? 2 : 1;
}

// ------------------------------------------------------------ tuning table
// Lines of `key=value` tokens, '#' starts a comment.  The first token is the
// entry kind (`moe` or `linear`); shape keys T (a value or a range lo-hi),
// k, E, H, I, K, N, L, r must match when present (absent = any); the choice
// keys tn (16/32/64/128/256), ksplit (1..4) and phases (1 = one launch per
// projection, 2 = both projections in one launch on single-CTA tiles)
// override the built-in choice.  The first matching line wins.
struct TuneEntry {
  bool linear = false;
  int t_lo = 0, t_hi = 0x7fffffff;
  int k = -1, E = -1, H = -1, I = -1, L = -1, r = -1;   // H = K, I = N for linear
  int tn = 0, ksplit = 0, phases = 0, guksplit = 0;
};

std::mutex g_tune_mu;
std::vector<TuneEntry> g_tune;

bool parse_tune_line(const std::string& line, TuneEntry& e, bool& is_entry) {
  std::string body = line.substr(0, line.find('#'));
  std::istringstream in(body);
  std::string tok;
  is_entry = false;
  if (!(in >> tok)) return true;   // blank
  if (tok == "moe") e.linear = false;
  else if (tok == "linear") e.linear = true;
  else return false;
  is_entry = true;
  while (in >> tok) {
    const size_t eq = tok.find('=');
    if (eq == std::string::npos) return false;
    const std::string key = tok.substr(0, eq), val = tok.substr(eq + 1);
    char* end = nullptr;
    if (key == "T") {
      // a value or lo-hi, both plain decimal numbers
      const size_t dash = val.find('-');
      const std::string lo = val.substr(0, dash);
      const std::string hi = dash == std::string::npos ? lo : val.substr(dash + 1);
      if (lo.empty() || hi.empty() || lo.size() > 9 || hi.size() > 9 ||
          lo.find_first_not_of("0123456789") != std::string::npos ||
          hi.find_first_not_of("0123456789") != std::string::npos)
        return false;
      e.t_lo = std::atoi(lo.c_str());
      e.t_hi = std::atoi(hi.c_str());
      if (e.t_hi < e.t_lo) return false;
      continue;
    }
    const long v = std::strtol(val.c_str(), &end, 10);
    if (!end || *end != '\0' || val.empty()) return false;
    const int iv = static_cast<int>(v);
    if (key == "k") e.k = iv;
    else if (key == "E") e.E = iv;
    else if (key == "H" || key == "K") e.H = iv;
    else if (key == "I" || key == "N") e.I = iv;
    else if (key == "L") e.L = iv;
    else if (key == "r") e.r = iv;
    else if (key == "tn") {
      if (iv != 16 && iv != 32 && iv != 64 && iv != 128 && iv != 256) return false;
      e.tn = iv;
    } else if (key == "ksplit") {
      if (iv < 1 || iv > 4) return false;
      e.ksplit = iv;
    } else if (key == "phases") {
      if (iv < 1 || iv > 2) return false;
      e.phases = iv;
    } else if (key == "guksplit") {
      if (iv < 1 || iv > 4) return false;
      e.guksplit = iv;
    } else {
      return false;
    }
  }
  return true;
}

int load_tune_file(const std::string& path, std::vector<TuneEntry>& out) {
  std::ifstream f(path);
  if (!f) return MOELORA_ERR_INVALID_ARG;
  std::string line;
  while (std::getline(f, line)) {
    TuneEntry e;
    bool is_entry = false;
    if (!parse_tune_line(line, e, is_entry)) return MOELORA_ERR_INVALID_ARG;
    if (is_entry) out.push_back(e);
  }
  return MOELORA_OK;
}

// Choice for a shape from the loaded table (tn, ksplit; 0 = no override).
void tune_lookup(bool linear, int T, int k, int E, int H, int I, int L, int r, int& tn, int& ks,
                 int* phases = nullptr, int* guksplit = nullptr) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  for (const TuneEntry& e : g_tune) {
    if (e.linear != linear || T < e.t_lo || T > e.t_hi) continue;
    if ((e.k >= 0 && e.k != k) || (e.E >= 0 && e.E != E) || (e.H >= 0 && e.H != H) ||
        (e.I >= 0 && e.I != I) || (e.L >= 0 && e.L != L) || (e.r >= 0 && e.r != r))
      continue;
    if (e.tn) tn = e.tn;
    if (e.ksplit) ks = e.ksplit;
    if (phases && e.phases) *phases = e.phases;
    if (guksplit && e.guksplit) *guksplit = e.guksplit;
    return;
  }
}

// LoRA ranks: multiples of 16 (the MMA's K step) up to 128 (one adapter's
// rows fill a 128-row shrink tile).
bool lora_rank_ok(int r) { return r >= 16 && r <= 128 && r % 16 == 0; }

// Width of one LoRA K chunk in shared memory: the largest of 64, 32, 16
// elements that divides r (a swizzle atom row of 128, 64 or 32 bytes).
uint32_t lora_chunk_width(int r) { return r % 64 == 0 ? 64u : (r % 32 == 0 ? 32u : 16u); }

int check_moe_dims(const moelora_dims* d) {
  if (!d) return MOELORA_ERR_INVALID_ARG;
  if (d->T < 0 || d->k < 1 || d->E < 1 || d->k > d->E || d->H < 8 || d->I < 8 || d->L < 0 ||
      d->r < 0)
    return MOELORA_ERR_INVALID_ARG;
  if (d->H % 8 || d->I % 8) return MOELORA_ERR_UNSUPPORTED;
  const bool lora = d->L > 0 && d->r > 0;
  if (lora && !lora_rank_ok(d->r)) return MOELORA_ERR_UNSUPPORTED;
  const int Lp = lora ? d->L + 1 : 1;
  if (d->E > kMaxExperts || static_cast<long long>(d->E) * Lp > kMaxBins)
    return MOELORA_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->T) * d->k >= (1ll << 30)) return MOELORA_ERR_UNSUPPORTED;
  return MOELORA_OK;
}

int check_linear_dims(const moelora_linear_dims* d) {
  if (!d) return MOELORA_ERR_INVALID_ARG;
  if (d->T < 0 || d->K < 8 || d->N < 8 || d->L < 0 || d->r < 0) return MOELORA_ERR_INVALID_ARG;
  if (d->K % 8 || d->N % 8) return MOELORA_ERR_UNSUPPORTED;
  const bool lora = d->L > 0 && d->r > 0;
  if (lora && !lora_rank_ok(d->r)) return MOELORA_ERR_UNSUPPORTED;
  if ((lora ? d->L + 1 : 1) > kMaxBins) return MOELORA_ERR_UNSUPPORTED;
  if (d->T >= (1 << 30)) return MOELORA_ERR_UNSUPPORTED;
  return MOELORA_OK;
}

// Align scratch common to every entry point.
void plan_align_scratch(Plan& p, Bump& b) {
  p.n = p.T * p.k;
  p.nbins = p.E * (p.L + 1);
  p.nchunks = (p.n + kAlignChunk - 1) / kAlignChunk;
  p.off_hdr = b.take(sizeof(WsHeader));
  p.off_chunk_hist = b.take(static_cast<size_t>(p.nchunks) * p.nbins * 4);
  p.off_bin_of = b.take(static_cast<size_t>(p.n) * 4);
  p.off_rank_of = b.take(static_cast<size_t>(p.n) * 4);
  p.off_bin_start = b.take(static_cast<size_t>(p.nbins) * 4);
}

// K splits of the shrink items.  A shrink item carries its slots' whole
// reduction (K = H or I) through the pipeline of one SM while the expand of
// every main item of its tile waits for it; on weight-streaming (unpaired)
// tiles that chain is latency-bound, and with a long K it outlasted the main
// items (E = 1, H = 8192, I = 14336, T = 8: the down phase took 105 us with
// whole-K shrink items, 53 us with 8 parts).  Split so that a part runs at
// most kShrinkStages pipeline stages; its fp32 part is summed in split order
// by the last part to finish.  CTA-pair (tensor-bound) tiles keep one part.
// MOELORA_SHRINK_SPLITS (1..8) overrides the choice.
constexpr int kShrinkStages = 8;

int choose_shrink_splits(const Plan& p) {
  if (!p.lora) return 1;
  const int kmin = p.linear ? p.H : std::min(p.H, p.I);
  const int kmax = p.linear ? p.H : std::max(p.H, p.I);
  int s;
  if (const int f = env_override("MOELORA_SHRINK_SPLITS", 1, 8)) {
    s = f;
  } else if (moe_gemm_paired(p.tn)) {
    s = 1;
  } else {
    const int kkb = moe_gemm_stage_kblocks(p.tn);
    const int stages = ((kmax + 63) / 64 + kkb - 1) / kkb;
    s = std::min(8, (stages + kShrinkStages - 1) / kShrinkStages);
  }
  // every part gets at least one K block of the shorter phase
  return std::max(1, std::min(s, (kmin + 63) / 64));
}

void plan_gemm_tables(Plan& p, Bump& b) {
  p.Pmax = p.n + p.E * (p.block_m - 1);
  // token tile: the smallest of 16/32/64/128/256 rows that holds an average
  // expert's rows (smaller tiles leave room for more pipeline stages)
  const int avg = (p.n + p.E - 1) / p.E;
  p.tn = avg <= 16 ? 16 : (avg <= 32 ? 32 : (avg <= 64 ? 64 : (avg <= 128 ? 128 : 256)));
  int t_tn = 0, t_ks = 0;
  tune_lookup(p.linear, p.T, p.k, p.E, p.H, p.linear ? p.N : p.I, p.L, p.r, t_tn, t_ks);
  if (t_tn) p.tn = t_tn;
  if (const int f = env_override("MOELORA_TN", 16, 256))
    if (f == 16 || f == 32 || f == 64 || f == 128 || f == 256) p.tn = f;
  // (a tile's L2 group is packed as first tile * 256 + length into one int,
  // so fewer than 2^23 tiles: 256-row tiles always give that, T * k < 2^30)
  if (static_cast<long long>(p.n) / p.tn + p.E + 1 >= (1ll << 23)) p.tn = 256;
  p.n_tiles_max = p.n / p.tn + std::min(p.E, std::max(p.n, 1)) + 1;
  p.n_slots_max = p.lora ? std::min(p.n, p.E * p.L + p.n_tiles_max) : 0;
  p.n_sh_max = p.n_slots_max;
  p.sks = choose_shrink_splits(p);
  p.off_row_tok = b.take(static_cast<size_t>(p.Pmax) * 4);
  p.off_row_w = b.take(static_cast<size_t>(p.Pmax) * 4);
  p.off_pos_of = b.take(static_cast<size_t>(p.n) * 4);
  p.off_tiles = b.take(static_cast<size_t>(p.n_tiles_max) * sizeof(TileInfo));
  p.off_shrink = b.take(static_cast<size_t>(std::max(p.n_sh_max, 1)) * p.sks * sizeof(ShrinkItem));
  p.off_sh_cnt = b.take(static_cast<size_t>(std::max(p.n_sh_max, 1)) * 2 * 4);
  p.off_slot_ad = b.take(static_cast<size_t>(std::max(p.n_slots_max, 1)) * 4);
  p.off_tile_done = b.take(static_cast<size_t>(p.n_tiles_max) * 4);
  p.off_act_done = b.take(static_cast<size_t>(p.n_tiles_max) * 4);
  p.off_xperm = b.take(static_cast<size_t>(p.Pmax) * p.H * 2);
  // gate_up shrink results: per slot and token row, hi and lo bf16 rows of r
  // (the dense linear uses the first half only)
  const size_t zbytes = static_cast<size_t>(p.n_slots_max) * p.tn * p.r * 2 * 2;
  p.off_zgu = b.take(std::max<size_t>(zbytes, 16));
  // fp32 parts of split shrink results [sks][slots * tn][r]
  if (p.sks > 1)
    p.off_zpart = b.take(static_cast<size_t>(p.sks) * p.n_slots_max * p.tn * p.r * 4);
}

// K splits for the last GEMM phase.  Decode-sized batches have few token
// tiles, so 128-row weight tiles alone give too few work items to fill the
// SMs in whole waves; splitting K (partials summed in order by the combine)
// multiplies the items.  Chosen from the sizes alone (workspace sizing must
// not depend on the device), for the 152 SMs of a GB300.
constexpr int kNominalSms = 152;

int choose_ksplit(double est_tiles, int n_mtiles, int K, double rows_per_expert) {
  if (const int f = env_override("MOELORA_KSPLIT", 1, 4)) return f;
  if (rows_per_expert > 64) return 1;            // tensor-bound: no split
  const int nk = (K + 63) / 64;
  if (nk / 2 < 16) return 1;                     // keep >= 16 K blocks per split
  const double items = std::max(1.0, est_tiles) * n_mtiles;
  if (items >= 8.0 * kNominalSms) return 1;      // enough items for a short tail
  auto eff = [](double n) { return n / (std::ceil(n / kNominalSms) * kNominalSms); };
  // two splits when that does not worsen the last wave (measured: more than
  // two splits costs more in partial traffic than it gains in balance)
  return eff(2 * items) >= eff(items) ? 2 : 1;
}

// K splits of the gate_up phase.  Its items cannot be split like the down
// phase's (the activation needs the whole sum), so a split writes its fp32
// part and the last split to arrive sums the parts and applies SiLU * up.
// Meant for layers whose gate_up phase has few items for the persistent
// grid (one expert: I / 64 weight tiles, 224 for I = 14336, 1.47 waves of
// 152 SMs).  Measured on the dense MLP (same box): T = 1 129.6 -> 127.4 us
// with 2 splits and two launches, T = 8 139.3 -> 137.3 us with 2 splits in
// the two-phase launch, T = 64 188.6 -> 200.0 us (worse: the summing split's
// epilogue holds its accumulator).  So the built-in choice is no split; the
// tuning table's `guksplit` key (or MOELORA_GU_KSPLIT) sets it per workload.
// Single-CTA tiles only, at least 16 K blocks per split.
int choose_gate_up_ksplit(int K, bool paired) {
  if (paired) return 1;
  const int nk = (K + 63) / 64;
  const int s = env_override("MOELORA_GU_KSPLIT", 1, 4);
  return std::max(1, std::min({s > 0 ? s : 1, 4, nk / 16}));
}

// K-block starts of the splits of a GEMM phase.  The main items are claimed
// split by split, so the last split's items are the ones a finishing SM
// takes last; from three splits up that split gets half the K blocks of the
// others, which shortens the idle tail at the end of the launch (the
// partials are summed the same way; measured on the dense linear: T = 64
// with 3 splits 114.8 -> 112.7 us, T = 8 with 4 splits 93.3 -> 92.8 us; with
// 2 splits it gained on one workload and lost on another, so those stay
// uniform).  Uniform splits also when K is too short.
void set_splits(GemmParams& g, int ksplit, int K, int bk) {
  const int nk = std::max(1, (K + bk - 1) / bk);
  g.ksplit = ksplit;
  const int weight_total = 2 * (ksplit - 1) + 1;
  bool ok = ksplit > 2 && nk >= 2 * weight_total;
  if (ok) {
    for (int i = 0; i <= ksplit; ++i)
      g.split_k0[i] = static_cast<int>((static_cast<long long>(nk) * std::min(2 * i, weight_total) +
                                        weight_total / 2) / weight_total);
    for (int i = 0; i < ksplit; ++i) ok = ok && g.split_k0[i + 1] > g.split_k0[i];
  }
  if (!ok) {
    const int per = (nk + ksplit - 1) / ksplit;
    for (int i = 0; i <= ksplit; ++i) g.split_k0[i] = std::min(nk, i * per);
  }
}

// Largest split count <= want for which every one of the splits of nk K
// blocks (ceil(nk / s) blocks each) is non-empty.
int clamp_ksplit(int want, int K) {
  const int nk = std::max(1, (K + 63) / 64);
  int s = std::max(1, std::min(want, nk));
  while (s > 1 && (s - 1) * ((nk + s - 1) / s) >= nk) --s;
  return s;
}

// Expected token tiles of a call: experts touched under uniform routing
// plus the extra tiles of experts with more than tn rows.
double expected_tiles(int T, int k, int E, int tn) {
  const double touched = E * (1.0 - std::pow(1.0 - static_cast<double>(k) / E, T));
  return std::floor(touched + 0.5) + std::floor(static_cast<double>(T) * k / tn);
}

Plan plan_forward(const moelora_dims* d) {
  Plan p;
  p.T = d->T; p.k = d->k; p.E = d->E; p.H = d->H; p.I = d->I;
  p.lora = d->L > 0 && d->r > 0;
  p.L = p.lora ? d->L : 0;
  p.r = p.lora ? d->r : 0;
  Bump b;
  plan_align_scratch(p, b);
  plan_gemm_tables(p, b);
  const size_t zbytes = static_cast<size_t>(p.n_slots_max) * p.tn * p.r * 2;   // one bf16 row
  p.off_zd = b.take(std::max<size_t>(zbytes, 16));
  p.off_act = b.take(static_cast<size_t>(p.Pmax) * p.I * 2);
  p.off_topk_ids = b.take(static_cast<size_t>(p.n) * 4);
  p.off_topk_w = b.take(static_cast<size_t>(p.n) * 4);
  p.ksplit = choose_ksplit(expected_tiles(p.T, p.k, p.E, p.tn), (p.H + 127) / 128, p.I,
                           static_cast<double>(p.n) / p.E);
  {
    int t_tn = 0, t_ks = 0;
    tune_lookup(false, p.T, p.k, p.E, p.H, p.I, p.L, p.r, t_tn, t_ks);
    if (t_ks && !env_override("MOELORA_KSPLIT", 1, 4)) p.ksplit = t_ks;
  }
  p.ksplit = clamp_ksplit(p.ksplit, p.I);
  p.off_ypair = b.take(static_cast<size_t>(p.ksplit) * p.Pmax * p.H * 4);
  p.gksplit = choose_gate_up_ksplit(p.H, moe_gemm_paired(p.tn));
  {
    int t_tn = 0, t_ks = 0, t_gks = 0;
    tune_lookup(false, p.T, p.k, p.E, p.H, p.I, p.L, p.r, t_tn, t_ks, nullptr, &t_gks);
    if (t_gks && !env_override("MOELORA_GU_KSPLIT", 1, 4) && !moe_gemm_paired(p.tn))
      p.gksplit = std::max(1, std::min(t_gks, ((p.H + 63) / 64) / 16));
  }
  if (p.gksplit > 1) {
    const size_t slots = static_cast<size_t>(p.n_tiles_max) * ((p.I + 63) / 64);
    p.off_gupart = b.take(static_cast<size_t>(p.gksplit) * slots * 128 * p.tn * 4);
    p.off_gucnt = b.take(slots * 4);
  }
  p.total = b.cur;
  return p;
}

Plan plan_linear(const moelora_linear_dims* d) {
  Plan p;
  p.linear = true;
  p.T = d->T; p.k = 1; p.E = 1; p.H = d->K; p.I = 0; p.N = d->N;
  p.lora = d->L > 0 && d->r > 0;
  p.L = p.lora ? d->L : 0;
  p.r = p.lora ? d->r : 0;
  Bump b;
  plan_align_scratch(p, b);
  plan_gemm_tables(p, b);
  p.ksplit = choose_ksplit(std::ceil(static_cast<double>(p.T) / p.tn), (p.N + 127) / 128, p.H,
                           static_cast<double>(p.T));
  {
    int t_tn = 0, t_ks = 0;
    tune_lookup(true, p.T, 1, 1, p.H, p.N, p.L, p.r, t_tn, t_ks);
    if (t_ks && !env_override("MOELORA_KSPLIT", 1, 4)) p.ksplit = t_ks;
  }
  p.ksplit = clamp_ksplit(p.ksplit, p.H);
  if (p.ksplit > 1)   // split partials in fp32, summed into out by the combine
    p.off_ypair = b.take(static_cast<size_t>(p.ksplit) * p.Pmax * p.N * 4);
  p.total = b.cur;
  return p;
}

Plan plan_align(const moelora_dims* d) {
  Plan p;
  p.T = d->T; p.k = d->k; p.E = d->E;
  p.L = d->L;   // the align keys on every adapter id in [-1, L)
  Bump b;
  plan_align_scratch(p, b);
  p.total = b.cur;
  return p;
}

// ------------------------------------------------------------ device info
int device_sms() {
  static std::mutex mu;
  static int cached_dev = -1;
  static int cached_sms = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(mu);
  if (dev != cached_dev) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached_dev = dev;
    cached_sms = sms;
  }
  return cached_sms;
}

// ------------------------------------------------------------ tensor maps
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

CUtensorMapSwizzle swizzle_for_bytes(int inner_bytes) {
  if (inner_bytes >= 128) return CU_TENSOR_MAP_SWIZZLE_128B;
  if (inner_bytes >= 64) return CU_TENSOR_MAP_SWIZZLE_64B;
  return CU_TENSOR_MAP_SWIZZLE_32B;
}

// bf16 tensor map; dims[0] is the contiguous axis; strides in elements of
// dims 1.. (converted to bytes here).
bool encode_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                const uint64_t* strides_elems, const uint32_t* box) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t gdim[5];
  cuuint64_t gstride[4];
  cuuint32_t bdim[5];
  cuuint32_t estr[5];
  for (int i = 0; i < rank; ++i) {
    gdim[i] = dims[i];
    bdim[i] = box[i];
    estr[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gstride[i] = strides_elems[i] * 2;
  const CUresult res = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), gdim,
                           gstride, bdim, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           swizzle_for_bytes(static_cast<int>(box[0]) * 2),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS;
}

bool enc2(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint32_t b0, uint32_t b1) {
  const uint64_t dims[2] = {d0, d1};
  const uint64_t str[1] = {d0};
  const uint32_t box[2] = {b0, b1};
  return encode_map(m, base, 2, dims, str, box);
}

bool enc3(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
          uint32_t b1) {
  const uint64_t dims[3] = {d0, d1, d2};
  const uint64_t str[2] = {d0, d0 * d1};
  const uint32_t box[3] = {b0, b1, 1};
  return encode_map(m, base, 3, dims, str, box);
}

// gate_up weight [E][2I][K] seen as (K, 2, I, E): one box brings 64
// features with each gate row followed by its up row (box row 2i = gate row
// i, 2i + 1 = up row i), so that the two accumulator rows of a feature land
// in adjacent TMEM lanes.
bool enc_gate_up(CUtensorMap* m, const void* base, uint64_t K, uint64_t I, uint64_t E, uint32_t bk) {
  const uint64_t dims[4] = {K, 2, I, E};
  const uint64_t str[3] = {I * K, K, 2 * I * K};
  const uint32_t box[4] = {bk, 2, 64, 1};
  return encode_map(m, base, 4, dims, str, box);
}

// gate_up LoRA expand weight [L][E][2I][r] seen as (r, 2, I, E, L), rows
// interleaved like the weight's.
bool enc_gate_up_lora(CUtensorMap* m, const void* base, uint64_t r, uint64_t I, uint64_t E,
                      uint64_t L, uint32_t box_w) {
  const uint64_t dims[5] = {r, 2, I, E, L};
  const uint64_t str[4] = {I * r, r, 2 * I * r, 2 * I * r * E};
  const uint32_t box[5] = {box_w, 2, 64, 1, 1};
  return encode_map(m, base, 5, dims, str, box);
}

bool enc4(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t d3,
          uint32_t b0, uint32_t b1, uint32_t b3 = 1) {
  const uint64_t dims[4] = {d0, d1, d2, d3};
  const uint64_t str[3] = {d0, d0 * d1, d0 * d1 * d2};
  const uint32_t box[4] = {b0, b1, 1, b3};
  return encode_map(m, base, 4, dims, str, box);
}

// token-operand and shrink-result maps for every box height up to tn
bool enc_row_maps(CUtensorMap* maps, const void* base, uint64_t width, uint64_t rows,
                  uint32_t box_w, int tn) {
  for (int i = 0; i < 5; ++i) {
    if ((16 << i) > tn) {
      std::memset(&maps[i], 0, sizeof(CUtensorMap));
      continue;
    }
    if (!enc2(&maps[i], base, width, rows, box_w, 16u << i)) return false;
  }
  return true;
}

// ------------------------------------------------------------ launch log / timing hook
std::mutex g_hook_mu;
cudaEvent_t g_events[64];
int g_n_events = 0;
int g_last_launches = 0;
const char* g_last_names[32];

struct Launcher {
  cudaStream_t stream;
  int count = 0;
  int n_events = 0;
  cudaEvent_t events[64];
  const char* names[32];
  explicit Launcher(cudaStream_t s) : stream(s) {
    std::lock_guard<std::mutex> lk(g_hook_mu);
    n_events = g_n_events;
    for (int i = 0; i < n_events; ++i) events[i] = g_events[i];
  }
  void before(const char* name) {
    if (count < n_events) cudaEventRecord(events[count], stream);
    if (count < 32) names[count] = name;
    ++count;
  }
  void finish() {
    if (count < n_events) cudaEventRecord(events[count], stream);
    std::lock_guard<std::mutex> lk(g_hook_mu);
    g_last_launches = count;
    for (int i = 0; i < count && i < 32; ++i) g_last_names[i] = names[i];
  }
};

// The align kernels (one kernel for small batches, which also clears the
// workspace error word; otherwise a memset does).  The single-CTA align is
// chained to whatever precedes it on the stream: it waits for that kernel's
// completion before its first read or write (a preceding call's combine may
// still be reading this workspace), so only its launch overlaps.
// With a.x set and no router, the small-batch align also gathers the token
// rows into x_perm when they total at most kFusedGatherBytes (measured: the
// decode batch's 368 KB and the dense T <= 8 rows gain ~0.8 us each; the
// dense T = 64 rows, 1 MB, lose 0.6 us against the separate permute);
// *gathered tells the caller whether it did.
constexpr size_t kFusedGatherBytes = 512 * 1024;

// L2 prefetch by extra CTAs of the small align (see align_prefetch) of the
// weights that the first GEMM phase streams first: its first routed
// experts' weight tiles in item order, the whole rows when the phase does
// not split K, else the first split's slice of each row.  Budgets measured
// on the GB300 with the prefetching CTAs starting before the preceding
// kernel ends (32 CTAs): whole experts 24 MB (decode 237.0 -> 234.8 us
// against none; 16 MB 235.3, 32 MB 237.3, 48 MB 236.1: more competes with the
// GEMM's own first loads), row slices 32 MB (dense T = 1 85.4 -> 83.0 us, T =
// 8 -> 87.7 us, dense MLP T = 1 -> 125.8 us; 64 MB slower).
// MOELORA_PF_MB / MOELORA_PF_CTAS override them (0 turns the prefetch off).
// The first phase: weight w, expert_bytes apart; rows of K bf16; weight tile
// m = feature rows [m * rows_per_m, +rows_per_m) and, for gate_up, the same
// rows up_rows further on; its first K split ends at K block k1 of bk.
void set_prefetch(AlignArgs& a, const void* w, long long expert_bytes, int K, int feat_rows,
                  int rows_per_m, long long up_rows, int n_m, int k1_blocks, int bk, bool ok) {
  a.pf_ctas = 0;
  const char* mb_env = std::getenv("MOELORA_PF_MB");
  const char* ct_env = std::getenv("MOELORA_PF_CTAS");
  const long long row_bytes = 2ll * K;
  const long long seg1 = std::min<long long>(K, static_cast<long long>(k1_blocks) * bk) * 2;
  const long long mb = mb_env ? std::atoll(mb_env) : (seg1 < row_bytes ? 32 : 24);
  const int ctas = ct_env ? std::atoi(ct_env) : 32;
  if (!ok || !w || mb <= 0 || ctas <= 0 || expert_bytes < 16 || seg1 < 16 || (seg1 & 15)) return;
  a.pf_base = static_cast<const unsigned char*>(w);
  a.pf_expert_bytes = expert_bytes & ~15ll;
  a.pf_bytes = mb << 20;
  a.pf_row_bytes = row_bytes;
  a.pf_seg0 = 0;
  a.pf_seg1 = seg1;
  a.pf_up_rows = up_rows;
  a.pf_rows_per_m = rows_per_m;
  a.pf_feat_rows = feat_rows;
  a.pf_n_m = n_m;
  a.pf_ctas = std::min(ctas, 64);
}

cudaError_t run_align(Launcher& ln, AlignArgs a, cudaStream_t stream, int num_sms, bool* gathered) {
  cudaError_t e;
  if (gathered) *gathered = false;
  if (a.x && static_cast<size_t>(a.n) * a.hv * 16 > kFusedGatherBytes) {
    a.x = nullptr;
    a.x_perm = nullptr;
  }
  if (a.n > 0 && align_small_fits(a)) {
    a.reset_err = 1;
    // rows gathered here: no permute reads the padding rows' tokens
    if (a.x && !a.logits) a.pad_rows = 0;
    ln.before("align_small");
    if ((e = launch_align_small(a, stream, true, num_sms)) != cudaSuccess) return e;
    if (gathered) *gathered = a.x != nullptr && a.logits == nullptr;
    return cudaSuccess;
  }
  if ((e = cudaMemsetAsync(&a.hdr->err, 0, sizeof(int), stream)) != cudaSuccess) return e;
  bool first = true;
  if (a.logits) {
    ln.before("route");
    if ((e = launch_route(a.logits, a.T, a.E, a.k, a.topk_ids_out, a.topk_w_out, stream, false)) !=
        cudaSuccess)
      return e;
    first = false;
  }
  if (a.nchunks > 0) {
    ln.before("align_hist");
    if ((e = launch_align_hist(a, stream, !first)) != cudaSuccess) return e;
    first = false;
  }
  ln.before("align_scan");
  if ((e = launch_align_scan(a, stream, !first)) != cudaSuccess) return e;
  if (a.nchunks > 0) {
    ln.before("align_scatter");
    if ((e = launch_align_scatter(a, stream, true)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Token tiles per L2 group of the main-item order (at most; a group is a run
// of one expert's tiles, and inside it the weight tile m is the slow index).
// The tiles of an expert then read each weight tile one after the other, and
// the run's token rows, at most ~16 MB of them, stay in L2 across all m.
int group_cap(int tn, int kmax) {
  if (const int f = env_override("MOELORA_GROUP_TILES", 1, 255)) return f;
  const double tile_bytes = static_cast<double>(tn) * kmax * 2.0;
  return static_cast<int>(std::max(1.0, std::min(255.0, std::floor(16.0 * (1 << 20) / tile_bytes))));
}

bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) != 0; }

template <typename T>
T* ws_ptr(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

AlignArgs align_args(const Plan& p, void* ws) {
  AlignArgs a;
  std::memset(&a, 0, sizeof(a));
  a.T = p.T; a.k = p.k; a.E = p.E; a.L = p.L;
  a.n = p.n; a.nbins = p.nbins; a.nchunks = p.nchunks;
  a.block_m = p.block_m; a.Pmax = p.Pmax;
  a.chunk_hist = ws_ptr<int>(ws, p.off_chunk_hist);
  a.bin_of = ws_ptr<int>(ws, p.off_bin_of);
  a.rank_of = ws_ptr<int>(ws, p.off_rank_of);
  a.bin_start = ws_ptr<int>(ws, p.off_bin_start);
  a.hdr = ws_ptr<WsHeader>(ws, p.off_hdr);
  return a;
}

void fill_gemm_tables(const Plan& p, void* ws, AlignArgs& a) {
  // the forward reads the rows' tokens, weights and positions and the GEMM
  // tables; the sorted order, block experts, segment offsets and row
  // adapters of the align entry point are not written
  a.sorted_ids = nullptr;
  a.blk_expert = nullptr;
  a.seg_off = nullptr;
  a.num_post_pad = nullptr;
  a.row_tok = ws_ptr<int>(ws, p.off_row_tok);
  a.row_lora = nullptr;
  a.pad_rows = 1;
  a.row_w = ws_ptr<float>(ws, p.off_row_w);
  a.pos_of = ws_ptr<int>(ws, p.off_pos_of);
  a.tn = p.tn;
  // a shrink item stacks up to 128 rows of adapters per CTA (two CTAs when
  // paired).  Unpaired (weight-streaming) tiles take fewer: a shrink item
  // then reads no more LoRA A bytes than a K-split main item reads weight
  // bytes, so the shrink items (which the main items' expand waits for) are
  // not the long pole -- with 8 adapters of r=16 over K=8192 one stacked
  // item streamed 2 MB while every main item streamed 1 MB.
  const bool paired = moe_gemm_paired(p.tn);
  // slots per shrink item: whole adapters per 128-row tile, on each CTA of a pair
  // (with split shrink items the parts are short anyway: full 128-row stacks,
  // which keep the number of items down -- the dense T = 64 linear with 8
  // parts of 2-slot items ran 122 us, with 8 parts of full stacks 116 us)
  a.spi = p.lora ? (paired ? 2 * (128 / p.r)
                           : (p.sks > 1 ? 128 / p.r : std::max(1, 128 / (p.r * p.ksplit))))
                 : 0;
  a.sks = p.sks;
  a.grp_max = group_cap(p.tn, std::max(p.H, p.I));
  a.tiles = ws_ptr<TileInfo>(ws, p.off_tiles);
  a.shrink = ws_ptr<ShrinkItem>(ws, p.off_shrink);
  a.sh_cnt = ws_ptr<int>(ws, p.off_sh_cnt);
  a.slot_adapter = ws_ptr<int>(ws, p.off_slot_ad);
  a.tile_done = ws_ptr<int>(ws, p.off_tile_done);
  a.gu_cnt = p.gksplit > 1 ? ws_ptr<int>(ws, p.off_gucnt) : nullptr;
  a.gu_nm = p.gksplit > 1 ? (p.I + 63) / 64 : 0;
}

// Spread a CTA-pair launch's shrink entries over its first K split (see the
// GEMM's item order) when its token rows, n rows of K bf16, are more than L2
// keeps across the launch's weight stream (measured on the GB300: the prefill
// batch's 94 MB of rows per projection, then read from DRAM once instead of
// twice; the skewed batch's 13 and 34 MB and the dense T = 512 linear's 8 MB
// gain nothing and lose 0.3-1% to the later shrink).
int spread_shrink(long long n_rows, int K) {
  if (const char* v = std::getenv("MOELORA_SPREAD_SHRINK")) return std::atoi(v) != 0 ? 1 : 0;
  return static_cast<double>(n_rows) * K * 2.0 > 64.0 * (1 << 20) ? 1 : 0;
}

GemmParams gemm_params(const Plan& p, void* ws, const AlignArgs& a) {
  GemmParams g;
  std::memset(&g, 0, sizeof(g));
  g.ksplit = 1;
  g.split_stride = 0;
  g.r = p.r;
  g.lora_w = p.lora ? static_cast<int>(lora_chunk_width(p.r)) : 64;
  g.lora_chunks = p.lora ? p.r / g.lora_w : 0;
  g.lora_swz = g.lora_w >= 64 ? 2 : (g.lora_w >= 32 ? 4 : 6);
  g.z_parts = 1;
  g.hdr = a.hdr;
  g.err = &a.hdr->err;
  g.tiles = a.tiles;
  g.shrink = a.shrink;
  g.slot_adapter = a.slot_adapter;
  g.row_lora = a.row_lora;
  g.bin_start = a.bin_start;
  g.lp1 = p.L + 1;
  g.row_w = a.row_w;
  g.row_tok = a.row_tok;
  g.tile_done = a.tile_done;
  g.Pmax = p.Pmax;
  g.T = p.T;
  g.n_experts = p.E;
  g.sh_splits = p.sks;
  g.zpart = p.sks > 1 ? ws_ptr<float>(ws, p.off_zpart) : nullptr;
  g.zpart_slots = p.n_slots_max;
  g.sh_cnt = a.sh_cnt;
  return g;
}

// Work units to launch: at most one per item (the launcher caps it at what
// can be resident at once).
int gemm_grid(const Plan& p, int n_mtiles, int sms) {
  (void)sms;
  const long long items = static_cast<long long>(p.n_sh_max) * p.sks +
                          static_cast<long long>(p.n_tiles_max) * n_mtiles;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(items, 1 << 20)));
}

#define MOELORA_CUDA_CHECK(expr)                 \
  do {                                           \
    if ((expr) != cudaSuccess) return MOELORA_ERR_CUDA; \
  } while (0)

}  // namespace

extern "C" {

size_t moelora_workspace_bytes(const moelora_dims* d) {
  if (check_moe_dims(d) != MOELORA_OK) return 0;
  return plan_forward(d).total;
}

size_t moelora_linear_workspace_bytes(const moelora_linear_dims* d) {
  if (check_linear_dims(d) != MOELORA_OK) return 0;
  return plan_linear(d).total;
}

size_t moelora_align_workspace_bytes(const moelora_dims* d) {
  if (!d || d->T < 0 || d->k < 1 || d->E < 1 || d->L < 0) return 0;
  if (d->E > kMaxExperts || static_cast<long long>(d->E) * (d->L + 1) > kMaxBins) return 0;
  return plan_align(d).total;
}

size_t moelora_align_capacity(const moelora_dims* d, int32_t block_m) {
  if (!d || d->T < 0 || d->k < 1 || d->E < 1 || block_m < 1 || block_m > 1024) return 0;
  return static_cast<size_t>(d->T) * d->k + static_cast<size_t>(d->E) * (block_m - 1);
}

int moe_lora_align(const moelora_dims* d, const int32_t* topk_ids, const int32_t* lora_ids,
                   int32_t block_m, int32_t* sorted_ids, int32_t* blk_expert, int32_t* seg_off,
                   int32_t* num_post_pad, void* ws, size_t ws_bytes, moelora_stream_t stream_) {
  if (!d || d->T < 0 || d->k < 1 || d->E < 1 || d->L < 0 || block_m < 1 || block_m > 1024)
    return MOELORA_ERR_INVALID_ARG;
  if (d->E > kMaxExperts || static_cast<long long>(d->E) * (d->L + 1) > kMaxBins)
    return MOELORA_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->T) * d->k >= (1ll << 30)) return MOELORA_ERR_UNSUPPORTED;
  if ((d->T > 0 && (!topk_ids || !lora_ids)) || !sorted_ids || !blk_expert || !seg_off ||
      !num_post_pad)
    return MOELORA_ERR_INVALID_ARG;
  if (!ws) return MOELORA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOELORA_ERR_MISALIGNED;
  const Plan p = plan_align(d);
  if (ws_bytes < p.total) return MOELORA_ERR_WORKSPACE;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  AlignArgs a = align_args(p, ws);
  a.topk_ids = topk_ids;
  a.lora_ids = lora_ids;
  a.block_m = block_m;
  a.Pmax = static_cast<int>(moelora_align_capacity(d, block_m));
  a.sorted_ids = sorted_ids;
  a.blk_expert = blk_expert;
  a.seg_off = seg_off;
  a.num_post_pad = num_post_pad;
  Launcher ln(stream);
  MOELORA_CUDA_CHECK(run_align(ln, a, stream, 0, nullptr));
  ln.finish();
  return MOELORA_OK;
}

}  // extern "C"

namespace {

// The forward, routed by topk_ids/topk_weights or, when logits is set, by the
// router run on device (fused into the align for small batches).
int forward_impl(const moelora_dims* d, const moelora_bf16* x, const int32_t* topk_ids,
                 const float* topk_weights, bool routed, const float* logits, const int32_t* lora_ids,
                 const moelora_bf16* W_gate_up, const moelora_bf16* W_down,
                 const moelora_bf16* A_gu, const moelora_bf16* B_gu, const moelora_bf16* A_d,
                 const moelora_bf16* B_d, moelora_bf16* out, void* ws, size_t ws_bytes,
                 moelora_stream_t stream_) {
  int st = check_moe_dims(d);
  if (st != MOELORA_OK) return st;
  if (routed && (d->k > 32 || d->E > kRouteMaxE)) return MOELORA_ERR_UNSUPPORTED;
  if (d->T == 0) return MOELORA_OK;
  const bool lora = d->L > 0 && d->r > 0;
  if (!x || (routed ? !logits : (!topk_ids || !topk_weights)) || !lora_ids || !W_gate_up ||
      !W_down || !out)
    return MOELORA_ERR_INVALID_ARG;
  if (lora && (!A_gu || !B_gu || !A_d || !B_d)) return MOELORA_ERR_INVALID_ARG;
  if (misaligned(x) || misaligned(W_gate_up) || misaligned(W_down) || misaligned(out))
    return MOELORA_ERR_MISALIGNED;
  if (lora && (misaligned(A_gu) || misaligned(B_gu) || misaligned(A_d) || misaligned(B_d)))
    return MOELORA_ERR_MISALIGNED;
  if (!ws) return MOELORA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOELORA_ERR_MISALIGNED;
  const Plan p = plan_forward(d);
  if (ws_bytes < p.total) return MOELORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MOELORA_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  AlignArgs a = align_args(p, ws);
  a.topk_ids = topk_ids;
  a.lora_ids = lora_ids;
  a.lora_ignore = p.lora ? 0 : 1;
  a.topk_weights = topk_weights;
  if (routed) {
    a.logits = logits;
    a.topk_ids_out = ws_ptr<int32_t>(ws, p.off_topk_ids);
    a.topk_w_out = ws_ptr<float>(ws, p.off_topk_w);
    a.topk_ids = a.topk_ids_out;
    a.topk_weights = a.topk_w_out;
  }
  fill_gemm_tables(p, ws, a);

  auto* x_perm = ws_ptr<__nv_bfloat16>(ws, p.off_xperm);
  auto* zgu = ws_ptr<__nv_bfloat16>(ws, p.off_zgu);
  auto* zd = ws_ptr<__nv_bfloat16>(ws, p.off_zd);
  auto* act = ws_ptr<__nv_bfloat16>(ws, p.off_act);
  auto* ypair = ws_ptr<float>(ws, p.off_ypair);
  const uint64_t zrows = static_cast<uint64_t>(std::max(p.n_slots_max, 1)) * p.tn;
  const uint32_t lw = p.lora ? lora_chunk_width(p.r) : 64u;

  // gate_up phase maps
  GemmMaps mg;
  std::memset(&mg, 0, sizeof(mg));
  const uint32_t bk = static_cast<uint32_t>(moe_gemm_kblock_width(p.tn));
  bool ok = enc_gate_up(&mg.w, W_gate_up, p.H, p.I, p.E, bk);
  ok = ok && enc_row_maps(mg.b, x_perm, p.H, p.Pmax, bk, p.tn);
  if (p.lora) {
    ok = ok && enc_gate_up_lora(&mg.lb, B_gu, p.r, p.I, p.E, p.L, lw);
    ok = ok && enc4(&mg.la, A_gu, p.H, p.r, p.E, p.L, bk, p.r);
    ok = ok && enc4(&mg.la_run, A_gu, p.H, p.r, p.E, p.L, bk, p.r, 128 / p.r);
    ok = ok && enc_row_maps(mg.z, zgu, 2 * p.r, zrows, lw, p.tn);
  }
  // down phase maps
  GemmMaps md;
  std::memset(&md, 0, sizeof(md));
  ok = ok && enc3(&md.w, W_down, p.I, p.H, p.E, bk, 128);
  ok = ok && enc_row_maps(md.b, act, p.I, p.Pmax, bk, p.tn);
  if (p.lora) {
    ok = ok && enc4(&md.lb, B_d, p.r, p.H, p.E, p.L, lw, 128);
    ok = ok && enc4(&md.la, A_d, p.I, p.r, p.E, p.L, bk, p.r);
    ok = ok && enc4(&md.la_run, A_d, p.I, p.r, p.E, p.L, bk, p.r, 128 / p.r);
    ok = ok && enc_row_maps(md.z, zd, p.r, zrows, lw, p.tn);
  }
  if (!ok) return MOELORA_ERR_CUDA;

  GemmParams gu = gemm_params(p, ws, a);
  gu.mode = kModeGateUp;
  gu.K = p.H;
  gu.spread_shrink = spread_shrink(p.n, gu.K);
  set_splits(gu, p.gksplit, gu.K, static_cast<int>(bk));
  if (p.gksplit > 1) {
    gu.gu_part = ws_ptr<float>(ws, p.off_gupart);
    gu.gu_cnt = a.gu_cnt;
    gu.gu_slots = p.n_tiles_max * ((p.I + 63) / 64);
  }
  const bool paired = moe_gemm_paired(p.tn);
  gu.n_mtiles = (p.I + (paired ? 127 : 63)) / (paired ? 128 : 64);
  gu.out_feats = p.I;
  gu.done_target = first_phase_done_target();
  gu.zbuf = zgu;
  gu.z_parts = 2;   // the gate_up shrink result as a bf16 hi/lo pair
  gu.out = act;
  gu.out_ld = p.I;
  gu.work_ctr = &a.hdr->work[0];

  GemmParams gd = gemm_params(p, ws, a);
  gd.mode = kModeDown;
  gd.K = p.I;
  gd.spread_shrink = spread_shrink(p.n, gd.K);
  gd.n_mtiles = (p.H + (paired ? 255 : 127)) / (paired ? 256 : 128);
  gd.out_feats = p.H;
  gd.done_target = 2;
  gd.zbuf = zd;
  gd.out = nullptr;
  gd.out_f32 = ypair;
  set_splits(gd, p.ksplit, gd.K, static_cast<int>(bk));
  gd.split_stride = static_cast<long long>(p.Pmax) * p.H;
  gd.out_ld = p.H;
  gd.work_ctr = &a.hdr->work[1];
  // the down phase's weights stream while the gate_up launch drains (measured:
  // decode 249.0 -> 246.4 us; on the gate_up and dense-linear launches, whose
  // predecessor is the short permute, the deferred first token rows cost more)
  gd.early_weights = 1;
  // Single-CTA tiles of a layer with several experts run both phases in
  // one persistent launch: a CTA that runs out of gate_up items goes on to
  // down items of tiles whose activations are complete, instead of idling
  // until the last gate_up item of the launch ends (decode 242.8 -> 239.0
  // us).  With one expert every down item waits for all of gate_up, and two
  // launches were as fast or faster (E = 1, T = 8: 146.0 against 152.3 us;
  // T = 64: 200.3 against 191.5, so the tuned table picks per workload).
  // The table's `phases` key or MOELORA_TWO_PHASE (0 / 1) override this.
  int phases = p.E > 1 ? 2 : 1;
  {
    int t_tn = 0, t_ks = 0;
    tune_lookup(false, p.T, p.k, p.E, p.H, p.I, p.L, p.r, t_tn, t_ks, &phases);
  }
  if (const char* tp = std::getenv("MOELORA_TWO_PHASE")) phases = std::strcmp(tp, "0") == 0 ? 1 : 2;
  const bool two_phase = !paired && phases == 2;
  if (two_phase) {
    int* act_done = ws_ptr<int>(ws, p.off_act_done);
    a.act_done = act_done;          // zeroed by the align
    gu.act_count = act_done;
    gd.act_wait = act_done;
    gd.act_target = gu.n_mtiles;   // one count per weight tile (the last K split's)
  }

  Launcher ln(stream);
  if (!routed) {   // the small-batch align gathers the token rows itself
    a.x = reinterpret_cast<const uint4*>(x);
    a.x_perm = reinterpret_cast<uint4*>(x_perm);
    a.hv = p.H / 8;
  }
  set_prefetch(a, W_gate_up, 2ll * p.I * p.H * 2, p.H, p.I, paired ? 128 : 64, p.I, gu.n_mtiles,
               gu.split_k0[1], static_cast<int>(bk), !routed);
  bool gathered = false;
  MOELORA_CUDA_CHECK(run_align(ln, a, stream, sms, &gathered));
  if (!gathered) {
    ln.before("permute");
    MOELORA_CUDA_CHECK(launch_permute(reinterpret_cast<const __nv_bfloat16*>(x), a.row_tok, x_perm,
                                      p.Pmax, p.H, p.T, &a.hdr->err, sms, stream));
  }
  if (two_phase) {
    ln.before("gemm_gate_up_down");
    MOELORA_CUDA_CHECK(launch_moe_gemm_two_phase(
        p.tn, mg, gu, md, gd, gemm_grid(p, gu.n_mtiles * p.gksplit + gd.n_mtiles * p.ksplit, sms),
        stream));
  } else {
    ln.before("gemm_gate_up");
    MOELORA_CUDA_CHECK(launch_moe_gemm(p.tn, mg, gu, gemm_grid(p, gu.n_mtiles * p.gksplit, sms), stream));
    ln.before("gemm_down");
    MOELORA_CUDA_CHECK(launch_moe_gemm(p.tn, md, gd, gemm_grid(p, gd.n_mtiles * p.ksplit, sms), stream));
  }
  ln.before("combine");
  MOELORA_CUDA_CHECK(launch_combine(ypair, a.pos_of, reinterpret_cast<__nv_bfloat16*>(out), p.T,
                                    p.k, p.H, p.ksplit, static_cast<long long>(p.Pmax) * p.H, p.Pmax,
                                    &a.hdr->err, sms, stream));
  ln.finish();
  return MOELORA_OK;
}

}  // namespace

extern "C" {

int moe_lora_forward(const moelora_dims* d, const moelora_bf16* x, const int32_t* topk_ids,
                     const float* topk_weights, const int32_t* lora_ids,
                     const moelora_bf16* W_gate_up, const moelora_bf16* W_down,
                     const moelora_bf16* A_gu, const moelora_bf16* B_gu, const moelora_bf16* A_d,
                     const moelora_bf16* B_d, moelora_bf16* out, void* ws, size_t ws_bytes,
                     moelora_stream_t stream) {
  return forward_impl(d, x, topk_ids, topk_weights, false, nullptr, lora_ids, W_gate_up, W_down,
                      A_gu, B_gu, A_d, B_d, out, ws, ws_bytes, stream);
}

int moe_lora_forward_routed(const moelora_dims* d, const moelora_bf16* x,
                            const float* router_logits, const int32_t* lora_ids,
                            const moelora_bf16* W_gate_up, const moelora_bf16* W_down,
                            const moelora_bf16* A_gu, const moelora_bf16* B_gu,
                            const moelora_bf16* A_d, const moelora_bf16* B_d, moelora_bf16* out,
                            void* ws, size_t ws_bytes, moelora_stream_t stream) {
  return forward_impl(d, x, nullptr, nullptr, true, router_logits, lora_ids, W_gate_up, W_down,
                      A_gu, B_gu, A_d, B_d, out, ws, ws_bytes, stream);
}

int moe_lora_route(const moelora_dims* d, const float* logits, int32_t* topk_ids,
                   float* topk_weights, moelora_stream_t stream) {
  if (!d || d->T < 0 || d->E < 1 || d->k < 1 || d->k > d->E) return MOELORA_ERR_INVALID_ARG;
  if (d->k > 32 || d->E > kRouteMaxE) return MOELORA_ERR_UNSUPPORTED;
  if (d->T == 0) return MOELORA_OK;
  if (!logits || !topk_ids || !topk_weights) return MOELORA_ERR_INVALID_ARG;
  Launcher ln(reinterpret_cast<cudaStream_t>(stream));
  ln.before("route");
  if (launch_route(logits, d->T, d->E, d->k, topk_ids, topk_weights,
                   reinterpret_cast<cudaStream_t>(stream), false) != cudaSuccess)
    return MOELORA_ERR_CUDA;
  ln.finish();
  return MOELORA_OK;
}

int moe_lora_linear(const moelora_linear_dims* d, const moelora_bf16* x, const int32_t* lora_ids,
                    const moelora_bf16* W, const moelora_bf16* A, const moelora_bf16* B,
                    moelora_bf16* out, void* ws, size_t ws_bytes, moelora_stream_t stream_) {
  int st = check_linear_dims(d);
  if (st != MOELORA_OK) return st;
  if (d->T == 0) return MOELORA_OK;
  const bool lora = d->L > 0 && d->r > 0;
  if (!x || !lora_ids || !W || !out) return MOELORA_ERR_INVALID_ARG;
  if (lora && (!A || !B)) return MOELORA_ERR_INVALID_ARG;
  if (misaligned(x) || misaligned(W) || misaligned(out) || (lora && (misaligned(A) || misaligned(B))))
    return MOELORA_ERR_MISALIGNED;
  if (!ws) return MOELORA_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) % kWsAlign) return MOELORA_ERR_MISALIGNED;
  const Plan p = plan_linear(d);
  if (ws_bytes < p.total) return MOELORA_ERR_WORKSPACE;
  const int sms = device_sms();
  if (sms <= 0) return MOELORA_ERR_CUDA;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);

  AlignArgs a = align_args(p, ws);
  a.topk_ids = nullptr;     // one expert
  a.lora_ids = lora_ids;
  a.lora_ignore = p.lora ? 0 : 1;
  a.topk_weights = nullptr; // weight 1
  fill_gemm_tables(p, ws, a);
  auto* x_perm = ws_ptr<__nv_bfloat16>(ws, p.off_xperm);
  auto* z = ws_ptr<__nv_bfloat16>(ws, p.off_zgu);
  const uint64_t zrows = static_cast<uint64_t>(std::max(p.n_slots_max, 1)) * p.tn;
  const uint32_t lw = p.lora ? lora_chunk_width(p.r) : 64u;

  GemmMaps m;
  std::memset(&m, 0, sizeof(m));
  const uint32_t bk = static_cast<uint32_t>(moe_gemm_kblock_width(p.tn));
  bool ok = enc3(&m.w, W, p.H, p.N, 1, bk, 128);
  ok = ok && enc_row_maps(m.b, x_perm, p.H, p.Pmax, bk, p.tn);
  if (p.lora) {
    ok = ok && enc4(&m.lb, B, p.r, p.N, 1, p.L, lw, 128);
    ok = ok && enc4(&m.la, A, p.H, p.r, 1, p.L, bk, p.r);
    ok = ok && enc4(&m.la_run, A, p.H, p.r, 1, p.L, bk, p.r, 128 / p.r);
    ok = ok && enc_row_maps(m.z, z, p.r, zrows, lw, p.tn);
  }
  if (!ok) return MOELORA_ERR_CUDA;

  GemmParams g = gemm_params(p, ws, a);
  g.K = p.H;
  g.spread_shrink = spread_shrink(p.n, g.K);
  const bool paired = moe_gemm_paired(p.tn);
  g.n_mtiles = (p.N + (paired ? 255 : 127)) / (paired ? 256 : 128);
  g.out_feats = p.N;
  g.done_target = first_phase_done_target();
  g.zbuf = z;
  g.out_ld = p.N;
  g.work_ctr = &a.hdr->work[0];
  set_splits(g, p.ksplit, g.K, static_cast<int>(bk));
  float* partial = p.ksplit > 1 ? ws_ptr<float>(ws, p.off_ypair) : nullptr;
  if (p.ksplit > 1) {
    // fp32 partial per K split (gate weight 1), summed by the combine
    g.mode = kModeDown;
    g.out_f32 = partial;
    g.split_stride = static_cast<long long>(p.Pmax) * p.N;
  } else {
    g.mode = kModeLinear;
    g.out = reinterpret_cast<__nv_bfloat16*>(out);
  }

  Launcher ln(stream);
  // the small-batch align gathers the token rows itself
  a.x = reinterpret_cast<const uint4*>(x);
  a.x_perm = reinterpret_cast<uint4*>(x_perm);
  a.hv = p.H / 8;
  set_prefetch(a, W, static_cast<long long>(p.N) * p.H * 2, p.H, p.N, paired ? 256 : 128, 0, g.n_mtiles,
               g.split_k0[1], static_cast<int>(bk), true);
  bool gathered = false;
  MOELORA_CUDA_CHECK(run_align(ln, a, stream, sms, &gathered));
  if (!gathered) {
    ln.before("permute");
    MOELORA_CUDA_CHECK(launch_permute(reinterpret_cast<const __nv_bfloat16*>(x), a.row_tok, x_perm,
                                      p.Pmax, p.H, p.T, &a.hdr->err, sms, stream));
  }
  ln.before("gemm_linear");
  MOELORA_CUDA_CHECK(launch_moe_gemm(p.tn, m, g, gemm_grid(p, g.n_mtiles * p.ksplit, sms), stream));
  if (p.ksplit > 1) {
    ln.before("combine");
    MOELORA_CUDA_CHECK(launch_combine(partial, a.pos_of, reinterpret_cast<__nv_bfloat16*>(out), p.T,
                                      1, p.N, p.ksplit, static_cast<long long>(p.Pmax) * p.N, p.Pmax,
                                      &a.hdr->err, sms, stream));
  }
  ln.finish();
  return MOELORA_OK;
}

int moe_lora_merge_adapter(const moelora_dims* d, int32_t adapter, const moelora_bf16* W_gate_up,
                           const moelora_bf16* W_down, const moelora_bf16* A_gu,
                           const moelora_bf16* B_gu, const moelora_bf16* A_d,
                           const moelora_bf16* B_d, moelora_bf16* W_gate_up_out,
                           moelora_bf16* W_down_out, moelora_stream_t stream_) {
  if (!d || d->E < 1 || d->H < 8 || d->I < 8 || d->L < 1 || d->r < 1) return MOELORA_ERR_INVALID_ARG;
  if (adapter < 0 || adapter >= d->L) return MOELORA_ERR_INVALID_ARG;
  if (!lora_rank_ok(d->r) || d->H % 8 || d->I % 8) return MOELORA_ERR_UNSUPPORTED;
  if (!W_gate_up || !W_down || !A_gu || !B_gu || !A_d || !B_d || !W_gate_up_out || !W_down_out)
    return MOELORA_ERR_INVALID_ARG;
  const void* ptrs[8] = {W_gate_up, W_down, A_gu, B_gu, A_d, B_d, W_gate_up_out, W_down_out};
  for (const void* q : ptrs)
    if (reinterpret_cast<uintptr_t>(q) % 16) return MOELORA_ERR_MISALIGNED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t E = d->E, H = d->H, I = d->I, r = d->r, a = adapter;
  auto bf = [](const moelora_bf16* p) { return reinterpret_cast<const __nv_bfloat16*>(p); };
  const uint32_t lw = lora_chunk_width(d->r);
  const int sms = device_sms();
  Launcher ln(stream);
  // adapter a's [E][...] slices are contiguous in the [L][E][...] LoRA tensors
  struct Proj {
    const char* name;
    const moelora_bf16* W;
    moelora_bf16* Wm;
    const moelora_bf16* B;
    const moelora_bf16* A;
    size_t rows, cols;
  };
  const Proj proj[2] = {
      {"merge_gate_up", W_gate_up, W_gate_up_out, B_gu + a * E * 2 * I * r, A_gu + a * E * r * H, 2 * I, H},
      {"merge_down", W_down, W_down_out, B_d + a * E * H * r, A_d + a * E * r * I, H, I}};
  for (const Proj& pj : proj) {
    CUtensorMap mw, mwm, mb;
    if (!enc3(&mw, pj.W, pj.cols, pj.rows, E, 64, 128) || !enc3(&mwm, pj.Wm, pj.cols, pj.rows, E, 64, 128) ||
        !enc3(&mb, pj.B, r, pj.rows, E, lw, 128))
      return MOELORA_ERR_CUDA;
    ln.before(pj.name);
    if (launch_merge(mw, mwm, mb, bf(pj.A), d->E, static_cast<int>(pj.rows), static_cast<int>(pj.cols),
                     d->r, sms, stream) != cudaSuccess)
      return MOELORA_ERR_CUDA;
  }
  ln.finish();
  return MOELORA_OK;
}

int moelora_load_tuning(const char* path) {
  std::vector<TuneEntry> table;
  if (path) {
    struct stat st;
    if (stat(path, &st) != 0) return MOELORA_ERR_INVALID_ARG;
    if (S_ISDIR(st.st_mode)) {
      // every *.cfg file of the folder, in name order
      DIR* dir = opendir(path);
      if (!dir) return MOELORA_ERR_INVALID_ARG;
      std::vector<std::string> names;
      while (dirent* de = readdir(dir)) {
        const std::string n = de->d_name;
        if (n.size() > 4 && n.compare(n.size() - 4, 4, ".cfg") == 0) names.push_back(n);
      }
      closedir(dir);
      std::sort(names.begin(), names.end());
      for (const std::string& n : names) {
        const int st2 = load_tune_file(std::string(path) + "/" + n, table);
        if (st2 != MOELORA_OK) return st2;
      }
    } else {
      const int st2 = load_tune_file(path, table);
      if (st2 != MOELORA_OK) return st2;
    }
  }
  std::lock_guard<std::mutex> lk(g_tune_mu);
  g_tune.swap(table);
  return MOELORA_OK;
}

int32_t moelora_tuning_entries(void) {
  std::lock_guard<std::mutex> lk(g_tune_mu);
  return static_cast<int32_t>(g_tune.size());
}

int moelora_set_timing_events(void* const* events, int32_t n_events) {
  if (n_events < 0 || n_events > 64 || (n_events > 0 && !events)) return MOELORA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lk(g_hook_mu);
  g_n_events = events ? n_events : 0;
  for (int i = 0; i < g_n_events; ++i) g_events[i] = static_cast<cudaEvent_t>(events[i]);
  return MOELORA_OK;
}

int32_t moelora_last_launch_count(void) {
  std::lock_guard<std::mutex> lk(g_hook_mu);
  return g_last_launches;
}

const char* moelora_last_launch_name(int32_t i) {
  std::lock_guard<std::mutex> lk(g_hook_mu);
  if (i < 0 || i >= g_last_launches || i >= 32) return "";
  return g_last_names[i];
}

int moelora_get_error(void* ws, moelora_stream_t stream) {
  if (!ws) return MOELORA_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return MOELORA_ERR_CUDA;
  int err = 0;
  if (cudaMemcpy(&err, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOELORA_ERR_CUDA;
  return err;
}

const char* moelora_status_string(int s) {
  switch (s) {
    case MOELORA_OK: return "ok";
    case MOELORA_ERR_INVALID_ARG: return "invalid argument";
    case MOELORA_ERR_UNSUPPORTED: return "unsupported size";
    case MOELORA_ERR_MISALIGNED: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case MOELORA_ERR_WORKSPACE: return "workspace missing or too small";
    case MOELORA_ERR_CUDA: return "CUDA error";
    case MOELORA_ERR_BAD_INDEX: return "expert or adapter id out of range";
    case MOELORA_ERR_TIMEOUT: return "a bounded device wait ran out";
    case MOELORA_ERR_DEVICE_CHECK: return "a device-side bounds check failed (checked build)";
    default: return "unknown status";
  }
}

}  // extern "C"
