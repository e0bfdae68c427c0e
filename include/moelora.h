/*
 * moelora.h -- C ABI of the GB300 (sm_103a) fused MoE-LoRA expert layer.
 *
 * What the layer computes (multi-LoRA MoE serving blog, vllm.com.cn/blog/
 * multi-lora, section "Implementing multi-LoRA for MoE in vLLM"):
 *   every token t carries k routed experts e_tj with gate weights w_tj and one
 *   adapter id a_t (-1 = no adapter).  For each routed pair
 *     g   = x W_gu[e]^T  + [a>=0] (x A_gu[a,e]^T) B_gu[a,e]^T     (y = xW + xAB)
 *     act = SiLU(g[:I]) * g[I:]
 *     d   = act W_d[e]^T + [a>=0] (act A_d[a,e]^T) B_d[a,e]^T
 *   and out[t] = sum_j w_tj d_tj (j ascending).  The page's W (h_in x h_out)
 *   is the transpose of the stored "out x in" matrices below; A is stored
 *   r x h_in and B h_out x r.  LoRA scale is 1; there is no bias.
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are DEVICE pointers on the current CUDA device;
 *    the caller owns all of them.  The library never allocates device
 *    memory: scratch lives in the caller's workspace (moe_lora_align_noalloc
 *    alone uses a fixed array of the library's own instead).
 *  - bf16 tensors are passed as moelora_bf16 (uint16_t bit patterns),
 *    row-major, the reduction axis contiguous, 16-byte aligned.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).  No entry point synchronises except moelora_get_error.
 *  - Return value: MOELORA_OK (0) or a negative MOELORA_ERR_* code.  Argument
 *    errors are reported before anything is enqueued.  Errors found by the
 *    kernels (bad ids, a bounded wait that ran out) are recorded in the
 *    workspace and read back with moelora_get_error.  Every wait in the
 *    kernels gives up after 2 s; the kernel then winds down and the next
 *    call runs normally.  A call whose wait ran out has still returned
 *    MOELORA_OK when it was enqueued; its output is undefined, and only
 *    moelora_get_error shows the MOELORA_ERR_TIMEOUT.  Setting the
 *    environment variable MOELORA_FAULT_INJECT=shrink_wait makes the first
 *    GEMM phase of each call wait for shrink results that never come, so that
 *    a test can see MOELORA_ERR_TIMEOUT.
 *  - The workspace needs no initialisation: every byte a call reads was
 *    written earlier in the same call.
 *  - Not thread-safe per workspace: two calls that share a workspace must be
 *    ordered on one stream.  Calls with separate workspaces may come from
 *    several host threads; the process-wide state is the tuning table and the
 *    timing hook (both guarded by a lock), a per-device cache of launch
 *    limits, filled on a device's first call (make one call per device before
 *    calling from several threads on different devices), and
 *    moe_lora_align_noalloc's scratch array with its device address, cached
 *    per device under a lock together with the id of the context it was
 *    found in (looked up again when that context has been replaced).
 */
#ifndef MOELORA_H_
#define MOELORA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moelora_bf16;           /* bf16 bit pattern */
typedef struct CUstream_st* moelora_stream_t;   /* == cudaStream_t */

enum {
  MOELORA_OK = 0,
  MOELORA_ERR_INVALID_ARG = -1,   /* null pointer, negative size, k > E ... */
  MOELORA_ERR_UNSUPPORTED = -2,   /* H, I not multiples of 8; r not a multiple of 16 in 16..128 */
  MOELORA_ERR_MISALIGNED = -3,    /* a bf16 pointer not 16-byte aligned */
  MOELORA_ERR_WORKSPACE = -4,     /* workspace null or smaller than required */
  MOELORA_ERR_CUDA = -5,          /* a CUDA runtime call or launch failed */
  MOELORA_ERR_BAD_INDEX = -6,     /* device: topk_ids / lora_ids out of range */
  MOELORA_ERR_TIMEOUT = -7,       /* device: a bounded wait ran out */
  MOELORA_ERR_DEVICE_CHECK = -8   /* device, checked builds only: an internal index
                                     failed its bounds check (the access was skipped) */
};

/* Sizes of one MoE-LoRA layer call.  T tokens, top-k, E experts, H hidden,
 * I intermediate (gate_up has 2I outputs), L adapter slots of rank r.
 * L == 0 or r == 0 means no LoRA at all (the adapter pointers may be NULL). */
typedef struct moelora_dims {
  int32_t T, k, E, H, I, L, r;
} moelora_dims;

/* Sizes of the dense multi-LoRA linear: x[T,K] W[N,K]^T + per-token LoRA. */
typedef struct moelora_linear_dims {
  int32_t T, K, N, L, r;
} moelora_linear_dims;

/* Bytes of device workspace moe_lora_forward needs for these sizes (host
 * only, no CUDA call).  Returns 0 for invalid sizes. */
size_t moelora_workspace_bytes(const moelora_dims* d);

/* Bytes of device workspace moe_lora_linear needs (host only). */
size_t moelora_linear_workspace_bytes(const moelora_linear_dims* d);

/* Bytes of device workspace moe_lora_align needs (host only). */
size_t moelora_align_workspace_bytes(const moelora_dims* d);

/* Capacity (entries) the sorted_ids buffer of moe_lora_align must have:
 * Pmax = T*k + E*(block_m - 1).  Host only; 0 for invalid sizes. */
size_t moelora_align_capacity(const moelora_dims* d, int32_t block_m);

/*
 * moe_lora_align -- group the T*k routed entries by (expert, adapter).
 *
 * Cited: multi-LoRA MoE blog, "Implementing multi-LoRA for MoE in vLLM" --
 * fused_moe runs one GEMM per expert over the tokens routed to it, and
 * fused_moe_lora adds one grid dimension over the active adapters; the
 * tokens are therefore grouped by expert and, inside an expert, by adapter.
 *
 * Definition (bit-exact contract): entry f = t*k + j has expert
 * e = topk_ids[t*k+j] and adapter a = lora_ids[t].  Entries are ordered by
 * the key (e, a+1, f); each expert's run is padded with the sentinel T*k to a
 * multiple of block_m (an expert with no entries gets no block).
 *   topk_ids_dev   [T*k] int32, in [0, E)
 *   lora_ids_dev   [T]   int32, in [-1, L); L may be 0 (all must be -1)
 *   block_m        padding granularity, 1..1024
 *   sorted_ids_dev [moelora_align_capacity] int32 out: positions [0, P) hold
 *                  the ordered entries and sentinels; [P, capacity) hold the
 *                  sentinel too
 *   blk_expert_dev [capacity / block_m] int32 out: expert of block b (< P/block_m)
 *   seg_off_dev    [E*(L+1)+1] int32 out: seg_off[e*(L+1)+a+1] = first position
 *                  of segment (e, a); seg_off[E*(L+1)] = P
 *   num_post_pad_dev [1] int32 out: P
 *   ws_dev, ws_bytes  scratch, at least moelora_align_workspace_bytes
 * Entries with an out-of-range id are left out of the order and flag
 * MOELORA_ERR_BAD_INDEX (read with moelora_get_error).
 */
int moe_lora_align(const moelora_dims* d, const int32_t* topk_ids_dev,
                   const int32_t* lora_ids_dev, int32_t block_m,
                   int32_t* sorted_ids_dev, int32_t* blk_expert_dev,
                   int32_t* seg_off_dev, int32_t* num_post_pad_dev,
                   void* ws_dev, size_t ws_bytes, moelora_stream_t stream);

/*
 * moe_lora_align_noalloc -- moe_lora_align without a workspace argument.
 *
 * The multi-LoRA MoE blog describes no such call: it exists for callers that cannot
 * allocate device memory -- code running while a stream is captured into a
 * CUDA graph (a cudaMalloc there breaks the capture), plug-ins handed
 * tensors but no allocator, and servers that reserved all device memory for
 * their own pool.  It computes exactly what moe_lora_align computes, with
 * the same inputs and outputs, but keeps its scratch in a fixed 4 MiB array
 * inside the library's device memory and allocates nothing.
 *   - Every GPU that loads the library holds those 4 MiB until process exit.
 *   - Sizes whose align scratch exceeds 4 MiB (about 256*(T*k/256+1)*E*(L+1)*4
 *     + 8*T*k + 4*E*(L+1) bytes) return MOELORA_ERR_WORKSPACE.
 *   - All calls share the one array: calls whose GPU work overlaps (on
 *     different streams without ordering) race; order them on one stream.
 *   - The first call on each device looks up the array's device address
 *     (and looks it up again once the device's context has been destroyed
 *     and created anew, as cudaDeviceReset does); make that call before any
 *     stream capture.
 *   - Out-of-range ids are left out of the order as in moe_lora_align, but
 *     the device error flag is not readable (there is no workspace to pass to
 *     moelora_get_error).
 */
int moe_lora_align_noalloc(const moelora_dims* d, const int32_t* topk_ids_dev,
                           const int32_t* lora_ids_dev, int32_t block_m,
                           int32_t* sorted_ids_dev, int32_t* blk_expert_dev,
                           int32_t* seg_off_dev, int32_t* num_post_pad_dev,
                           moelora_stream_t stream);

/*
 * moe_lora_forward -- the fused MoE-LoRA expert layer (formula at the top).
 *
 * Cited: multi-LoRA MoE blog, "Implementing multi-LoRA for MoE in vLLM"
 * (expert FFN = gate_up then down; y = xW + xAB with shrink z = xA and expand
 * zB; four LoRA operations per expert per adapter; expert outputs aggregated
 * with the router weights).
 *   x_dev            [T][H] bf16
 *   topk_ids_dev     [T][k] int32 in [0, E)
 *   topk_weights_dev [T][k] fp32 (used as given)
 *   lora_ids_dev     [T] int32 in [-1, L)
 *   W_gate_up_dev    [E][2I][H] bf16 (rows 0..I-1 gate, I..2I-1 up)
 *   W_down_dev       [E][H][I] bf16
 *   A_gu_dev [L][E][r][H], B_gu_dev [L][E][2I][r],
 *   A_d_dev  [L][E][r][I], B_d_dev  [L][E][H][r]   bf16 (NULL when no LoRA)
 *   out_dev          [T][H] bf16 out (fp32 accumulation, one rounding)
 *   ws_dev, ws_bytes scratch of at least moelora_workspace_bytes(d)
 * T == 0 is a successful no-op.  Outputs are deterministic: the same inputs
 * give bit-identical results.  Nothing is allocated and nothing synchronises,
 * so the call can be captured in a CUDA graph.
 */
int moe_lora_forward(const moelora_dims* d, const moelora_bf16* x_dev,
                     const int32_t* topk_ids_dev, const float* topk_weights_dev,
                     const int32_t* lora_ids_dev, const moelora_bf16* W_gate_up_dev,
                     const moelora_bf16* W_down_dev, const moelora_bf16* A_gu_dev,
                     const moelora_bf16* B_gu_dev, const moelora_bf16* A_d_dev,
                     const moelora_bf16* B_d_dev, moelora_bf16* out_dev,
                     void* ws_dev, size_t ws_bytes, moelora_stream_t stream);

/*
 * moe_lora_route -- the router step upstream of the layer: each token's
 * top-k experts and gate weights from its router logits.
 * Cited: multi-LoRA MoE blog, "Implementing multi-LoRA for MoE in vLLM" (the
 * routing algorithm sends each token to its most relevant experts and their
 * outputs are aggregated).
 * Definition: p = softmax(logits[t]); the k largest p are chosen, larger
 * first, the lower expert index first among equal logits (the choice is made
 * on the fp32 logits themselves); weights = p renormalised over the chosen k
 * (= softmax of the chosen logits), computed in fp32.
 *   logits_dev        [T][E] fp32
 *   topk_ids_dev      [T][k] int32 out
 *   topk_weights_dev  [T][k] fp32 out
 * Only d->T, d->k, d->E are read; k <= 32 and E <= 1024 (else
 * MOELORA_ERR_UNSUPPORTED).  No workspace.
 */
int moe_lora_route(const moelora_dims* d, const float* logits_dev, int32_t* topk_ids_dev,
                   float* topk_weights_dev, moelora_stream_t stream);

/*
 * moe_lora_forward_routed -- moe_lora_forward with the router step fused in:
 * takes router logits [T][E] (fp32) instead of topk_ids / topk_weights and
 * routes on the device (inside the single-CTA align for batches of up to
 * 1024 routed entries, as a separate kernel before the align above that).
 * Same workspace as moe_lora_forward (moelora_workspace_bytes); k <= 32,
 * E <= 1024.  The result is bit-identical to moe_lora_route followed by
 * moe_lora_forward on the same inputs.
 */
int moe_lora_forward_routed(const moelora_dims* d, const moelora_bf16* x_dev,
                            const float* router_logits_dev, const int32_t* lora_ids_dev,
                            const moelora_bf16* W_gate_up_dev, const moelora_bf16* W_down_dev,
                            const moelora_bf16* A_gu_dev, const moelora_bf16* B_gu_dev,
                            const moelora_bf16* A_d_dev, const moelora_bf16* B_d_dev,
                            moelora_bf16* out_dev, void* ws_dev, size_t ws_bytes,
                            moelora_stream_t stream);

/*
 * moe_lora_linear -- dense multi-LoRA linear, the one-expert, top-1,
 * weight-1 degenerate case of the layer with a single projection and no
 * activation: y[t] = x[t] W^T + [a_t>=0] (x[t] A[a_t]^T) B[a_t]^T.
 * Cited: same page and section (y = xW + xAB; existing dense multi-LoRA
 * kernels are the expert-free case).
 *   x_dev [T][K] bf16, lora_ids_dev [T] int32 in [-1, L),
 *   W_dev [N][K] bf16, A_dev [L][r][K] bf16, B_dev [L][N][r] bf16,
 *   out_dev [T][N] bf16 out, ws of at least moelora_linear_workspace_bytes.
 */
int moe_lora_linear(const moelora_linear_dims* d, const moelora_bf16* x_dev,
                    const int32_t* lora_ids_dev, const moelora_bf16* W_dev,
                    const moelora_bf16* A_dev, const moelora_bf16* B_dev,
                    moelora_bf16* out_dev, void* ws_dev, size_t ws_bytes,
                    moelora_stream_t stream);

/*
 * moe_lora_merge_adapter -- the merged-weight fast path for batches served by
 * a single adapter: writes W' = W + B A for adapter `adapter` and every
 * expert, both projections:
 *   W_gate_up_out[e] = W_gate_up[e] + B_gu[a][e] A_gu[a][e]   ([2I][H])
 *   W_down_out[e]    = W_down[e]    + B_d[a][e]  A_d[a][e]    ([H][I])
 * (fp32 accumulation, one bf16 rounding).  moe_lora_forward with L = 0 on the
 * merged weights then gives the LoRA layer for tokens of that adapter with no
 * shrink/expand work: x(W + AB) = xW + xAB.
 * Cited: the hybrid-attention decoder page, "static LoRA merge"
 * (merge_and_unload at initialisation removes the LoRA cost at run time), and
 * the multi-LoRA MoE blog's y = xW + xAB.
 *   d: E, H, I, L, r (T and k unused); 0 <= adapter < L; r a multiple of
 *   16 up to 128 and H, I multiples of 8 (else MOELORA_ERR_UNSUPPORTED);
 *   every pointer 16-byte aligned (else MOELORA_ERR_MISALIGNED).
 *   Outputs are caller-owned device buffers shaped like the inputs; they may
 *   not alias the inputs.  Run once per adapter switch; no workspace.  The
 *   rank-r products run on the tensor cores; the call moves each weight once
 *   in and once out (HBM-bound).  Its waits are bounded like the layer's,
 *   but with no workspace a wait that ran out cannot be reported (the merged
 *   weights are then undefined); none of its waits depends on another CTA.
 */
int moe_lora_merge_adapter(const moelora_dims* d, int32_t adapter,
                           const moelora_bf16* W_gate_up_dev, const moelora_bf16* W_down_dev,
                           const moelora_bf16* A_gu_dev, const moelora_bf16* B_gu_dev,
                           const moelora_bf16* A_d_dev, const moelora_bf16* B_d_dev,
                           moelora_bf16* W_gate_up_out_dev, moelora_bf16* W_down_out_dev,
                           moelora_stream_t stream);

/*
 * moelora_load_tuning -- load a table of tuned launch choices (host only).
 * Cited: multi-LoRA MoE blog, "Kernel config tuning" (block sizes and split
 * factors tuned per workload, loaded by users from a folder of config files).
 * `path` is a file or a folder (every *.cfg file in it, in name order); NULL
 * clears the table.  Each line: `moe` or `linear`, then key=value tokens;
 * shape keys T (value or range lo-hi), k, E, H, I (linear: K, N), L, r must
 * match when present; choice keys tn (token tile 16/32/64/128/256),
 * ksplit (1..4, K splits of the down / linear phase), phases (1: one launch
 * per projection, 2: both in one launch, single-CTA tiles) and guksplit
 * (1..4, K splits of the gate_up phase on single-CTA tiles, whose fp32 parts
 * the last split to arrive sums in split order) override the built-in
 * choice; the first matching line wins; '#' starts a comment.  Workspace
 * sizes depend on the choice: load the table before sizing workspaces.
 * Returns MOELORA_ERR_INVALID_ARG for a missing path or a malformed line
 * (the previous table is then kept).
 */
int moelora_load_tuning(const char* path);

/* Number of entries in the loaded tuning table (host only). */
int32_t moelora_tuning_entries(void);

/* Per-kernel timing hook: when `events` is non-NULL, the next calls record
 * events[i] (cudaEvent_t, created by the caller) on the call's stream before
 * launch i of the call and events[n_launches] after the last launch, for as
 * long as the hook is installed.  n_events is the array's length; launches
 * beyond it are not bracketed.  Pass NULL to remove.  Host only. */
int moelora_set_timing_events(void* const* events, int32_t n_events);

/* Number of kernel launches the last moe_lora_forward / moe_lora_linear call
 * made (host-side count; memset nodes are not counted). */
int32_t moelora_last_launch_count(void);

/* Name of the kernel launched as launch i of the last call (for reports). */
const char* moelora_last_launch_name(int32_t i);

/* Synchronises `stream`, returns the device-flagged status of the last call
 * that used this workspace (MOELORA_OK, _BAD_INDEX or _TIMEOUT), or
 * MOELORA_ERR_CUDA if the synchronisation itself failed. */
int moelora_get_error(void* ws_dev, moelora_stream_t stream);

/* Static text for a status code. */
const char* moelora_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* MOELORA_H_ */
