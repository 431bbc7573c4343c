/*
 * ftmoe.h - C ABI of the routed mixture-of-experts layer forward on B300 (sm_103a).
 *
 * The layer follows the FreeToken pages' statement of the problem:
 *   - a small router selects a few experts per token, e.g. 6 of 256
 *     (banandre.com, "The 284B Model on a 32GB GPU Trick", section
 *     "Sparsity Is a Lie (But a Useful One)");
 *   - resident experts run on GPU tensor cores from expert slots, with weights
 *     in MXFP4, NVFP4, FP8 or BF16 (zubnet.ai, "FreeToken, Unsloth GGUF ...
 *     consumer hardware");
 *   - partial sums over a split of the selected experts add up exactly once the
 *     layer completes (banandre.com, same page, section "The q* Policy: Math
 *     Instead of Guesses");
 *   - a global LRU over all MoE layers, which admits every missed expert,
 *     decides which experts are resident (asapai.co.kr, "Running 753B GLM-5.2
 *     on a single workstation GPU", section "Abandoning fixed offloading in
 *     favor of measured bandwidth"; banandre.com, section "Semantic-Aware
 *     Caching").
 *
 * Conventions for every call
 *   - Pointers are DEVICE pointers unless a parameter says "host".  The caller
 *     owns all memory.  The library never allocates or frees caller memory.
 *   - Scratch is passed as (ws, ws_bytes).  Its size comes from the matching
 *     *_workspace_size query.  Before its first use, the workspace's first
 *     FTMOE_WS_ZERO_BYTES bytes must be zero.  They hold the library's
 *     completion and grid-sync counters from call to call: the caller must not
 *     write them afterwards, except to zero them again after a call reported
 *     FTMOE_ERR_TIMEOUT.  One workspace must not be used by two calls that can
 *     run at the same time.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it.  Kernels are launched with programmatic dependent
 *     launch, so consecutive calls on one stream overlap their launch latency.
 *   - Layouts are row-major and contiguous.  bf16 values travel as uint16_t
 *     bit patterns.
 *   - Argument errors are found on the host before any launch, and return
 *     FTMOE_ERR_INVALID_ARG without touching memory.  Data errors found on the
 *     device (an id or slot out of range) never trap.  They set a device error
 *     word, which ftmoe_get_device_error reads and clears; the offending item
 *     is skipped.
 */
#ifndef FTMOE_H
#define FTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FTMOE_WS_ZERO_BYTES 256

typedef enum {
  FTMOE_OK = 0,
  FTMOE_ERR_INVALID_ARG = 1,   /* bad pointer, size or descriptor (host check) */
  FTMOE_ERR_UNSUPPORTED = 2,   /* valid request the library does not implement */
  FTMOE_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  FTMOE_ERR_WORKSPACE = 4,     /* ws_bytes below the *_workspace_size answer */
  FTMOE_ERR_TIMEOUT = 5,       /* a bounded device wait gave up */
  FTMOE_ERR_DEVICE_CHECK = 6   /* a device-side data check failed */
} ftmoe_status;

/* Expert weight storage formats.  K is the reduction dim, innermost in memory.
 *   BF16      w = bf16 value
 *   NVFP4     E2M1 codes, 2 per byte (element 2i = low nibble), one E4M3 scale
 *             per 16 consecutive K elements [N][K/16], one fp32 scale per tensor:
 *             w = e2m1 * e4m3 * tensor_scale
 *   MXFP4     E2M1 codes as above, one E8M0 scale per 32 K elements [N][K/32]:
 *             w = e2m1 * 2^(e8m0 - 127)
 *   FP8_B128  E4M3 codes [N][K], one fp32 scale per 128x128 block [N/128][K/128]:
 *             w = e4m3 * scale
 */
typedef enum { FTMOE_BF16 = 0, FTMOE_NVFP4 = 1, FTMOE_MXFP4 = 2, FTMOE_FP8_B128 = 3 } ftmoe_wfmt;

/* One MoE layer: E routed experts, top-k, model width d, expert width ffn. */
typedef struct {
  int E;        /* 1..1024 */
  int k;        /* 1..min(E, 32) */
  int d;        /* multiple of 256 */
  int ffn;      /* multiple of 128 */
  int fmt;      /* ftmoe_wfmt of the expert weights */
  int renorm;   /* 1: the k weights are divided by their sum; 0: raw softmax probabilities */
} ftmoe_layer_desc;

/* Expert weights of C slots (the slot arena).  Slot s of each array starts
 * at s times the per-slot size of that array:
 *   gate, up      [C][ffn][d]  codes (bf16: uint16; FP4: d/2 bytes per row; FP8: d bytes)
 *   down          [C][d][ffn]  codes
 *   *_scale       NVFP4: uint8 E4M3 [C][N][K/16]; MXFP4: uint8 E8M0 [C][N][K/32];
 *                 FP8_B128: float [C][N/128][K/128]; BF16: NULL
 *   tensor_scale  NVFP4: float [C][3] (gate, up, down); otherwise NULL
 * Every pointer must be 16-byte aligned. */
typedef struct {
  int fmt;
  int C;
  int d;
  int ffn;
  const void* gate;
  const void* up;
  const void* down;
  const void* gate_scale;
  const void* up_scale;
  const void* down_scale;
  const float* tensor_scale;
  /* Layouts derived by ftmoe_prepare_weights, or NULL.  Required when
   * ftmoe_expert_ffn_path reports 1 for the call (NVFP4 prefill); the decode
   * path of NVFP4 / MXFP4 runs faster with it. */
  const void* prepared;
} ftmoe_weights;

/* ---------------------------------------------------------------------------
 * ftmoe_prepare_weights - derived layouts of a slot arena that the fast kernels
 * read.  Run once per arena (or after slots are refilled), outside any timed
 * region.  The canonical arena stays the interchange format.  Up to three parts,
 * in this order in prep:
 *   1. Prefill (NVFP4, d and ffn multiples of 256): the weight block scales
 *      repacked for the tensor-core path.  Each MMA with K = 64 reads four scales
 *      per row from tensor memory; per 128 weight rows and per K = 64 step the
 *      layout holds the 512 bytes that fill four tensor-memory columns there: byte
 *      (r % 32) * 16 + (r / 32) * 4 + kb for row r of the 128 and 16-element
 *      block kb of the 64.  The tensor-core path reads the codes in place.
 *        gate/up  [C][ffn/NH][d/64][A][512]: an N tile of NH = 128 gate rows then
 *                 NH up rows in A = 2 blocks of 128 rows
 *        down     [C][d/128][ffn/64][512]
 *   2. Decode (NVFP4, MXFP4), starting at the next 1024-byte boundary: a copy of
 *      codes and scales in tiles that each stream into shared memory with one
 *      bulk copy, ordered so that warp-level MMA fragments read them without bank
 *      conflicts.  Per slot: ffn/16 gate/up tiles then d/32 down tiles.  A tile of
 *      R rows of one matrix holds its codes as [K/32][R][16 bytes] and its scales
 *      as [K/16 or K/32][R]; a gate/up tile is [gate codes][up codes][gate
 *      scales][up scales] (R = 16), a down tile [codes][scales] (R = 32).  Its
 *      size equals the canonical bytes of the slot.  Without it (weights->prepared
 *      NULL) the decode path reads the canonical arena, more slowly.
 *   3. Down slices (NVFP4, MXFP4, d <= 2048), right after part 2: for the layer
 *      call's slice form, per slot and per 16 columns n0 of W_down (ffn/16
 *      slices of 9*d bytes): the codes of W_down[:, 16 n0 .. 16 n0 + 16) as
 *      [d/16 row tiles][32 lanes][4 bytes], lane (g, t) holding bytes 2t and
 *      2t + 1 of rows g and g + 8 of the tile (the fragment a warp-level MMA
 *      reads), then one scale byte per row [d] (the block scale covering those 16
 *      columns).
 * weights->prepared is ignored here.  prep (device, prep_bytes from
 * ftmoe_prepare_weights_size, 256-byte aligned) is written; it is then passed as
 * weights->prepared.  BF16 and FP8_B128 need nothing: size 0, and the call
 * returns FTMOE_OK without work.
 * ------------------------------------------------------------------------- */
size_t ftmoe_prepare_weights_size(const ftmoe_layer_desc* desc, int C);
ftmoe_status ftmoe_prepare_weights(const ftmoe_layer_desc* desc, const ftmoe_weights* weights, void* prep,
                                   size_t prep_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * a1  ftmoe_route - router logits, top-k ids and their weights.
 * Pages: a small router selects a few experts for each token
 * (banandre.com, "The 284B Model on a 32GB GPU Trick", section "Sparsity Is a
 * Lie (But a Useful One)").  Reading: softmax over all E logits, then top-k;
 * ties go to the lower id.
 *   x          bf16 [T][d]
 *   w_router   bf16 [E][d]
 *   logit_bias fp32 [E] or NULL (added after the dot product)
 *   topk_ids   int32 [T][k]: ordered by (logit desc, id asc)
 *   topk_w     fp32 [T][k]: softmax probability of each chosen expert,
 *              divided by their sum when desc->renorm
 *   logits     fp32 [T][E] or NULL
 * The fp32 logit has one fixed definition (order R), so the ids are
 * reproducible bit for bit:
 *   - Chunk c = elements 8c..8c+7 belongs to lane c % 32.
 *   - Each lane sums its products in ascending element order from 0.0f.
 *     Each product is exact; each add is rounded to fp32.
 *   - The 32 lane sums combine by an xor butterfly over offsets 16, 8, 4, 2, 1.
 *   - The bias is added last.
 * Long batches (logits NULL, T >= 256, desc->renorm, E a multiple of 16 in
 * 16..256, d <= 4096) run the logits on tcgen05 tensor cores.  A per-token
 * error bound (relative 2 * (d/16 * 2^-22 + (d/32 + 5) * 2^-24) of
 * ||x|| max_e ||w_e||) keeps as candidates the experts within the bound of the
 * k-th value; their logits are recomputed in order R and the top-k taken from
 * them, so ids and weights equal those above bit for bit.  Tokens with more
 * than 32 candidates are recomputed entirely in order R.  The workspace's
 * uint32 at byte 128 then counts those tokens, and the uint32 at byte 132 the
 * tokens with more than k candidates.
 * Preconditions: 1 <= T <= 2^20, d % 256 == 0.
 * ------------------------------------------------------------------------- */
size_t ftmoe_route_workspace_size(const ftmoe_layer_desc* desc, int T);
ftmoe_status ftmoe_route(const ftmoe_layer_desc* desc, const uint16_t* x, const uint16_t* w_router,
                         const float* logit_bias, int T, int32_t* topk_ids, float* topk_w, float* logits,
                         void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * ftmoe_route_noalloc - ftmoe_route for callers that cannot allocate device memory.
 * The pages have no counterpart: this is a deployment convenience of this library.
 * Some callers cannot call cudaMalloc or own a workspace.  Examples: code running
 * under a memory pool that already owns the whole device budget, and code inside
 * another library's callback where an allocation could fail or synchronise the
 * device at an unpredictable moment.  This variant takes inputs and outputs only,
 * exactly as ftmoe_route does with logits = NULL.  Its scratch (a counter and the
 * [T][E] fp32 logits) is a fixed array inside the library that every GPU loading
 * it holds until the process exits; it allocates nothing and calls no allocating
 * routine.
 *   - T * E must not exceed FTMOE_NOALLOC_MAX_LOGITS (1 MiB of logits); larger
 *     requests return FTMOE_ERR_WORKSPACE.
 *   - The first call on a device looks up the array's device address (and the first
 *     call after a device reset, which ends the context the address belonged to).  Make
 *     that first call before capturing a stream.
 *   - All calls share the one array: calls that can overlap on the GPU (other
 *     streams, other host threads) race and must be serialised by the caller.
 * ------------------------------------------------------------------------- */
#define FTMOE_NOALLOC_MAX_LOGITS 262144
ftmoe_status ftmoe_route_noalloc(const ftmoe_layer_desc* desc, const uint16_t* x, const uint16_t* w_router,
                                 const float* logit_bias, int T, int32_t* topk_ids, float* topk_w, void* stream);

/* ---------------------------------------------------------------------------
 * a3  ftmoe_quantize_act - the prefill activation quantiser on its own.
 * The pages do not say how activations reach FP4 / FP8 tensor cores.  The
 * library's rules, applied inside ftmoe_expert_ffn's tensor-core paths to the
 * gathered rows of x (and to h), by the layer's weight format:
 *   NVFP4     per block of 16 consecutive elements of a row:
 *               s_code = E4M3_rn_satfinite(amax / 6)            (IEEE fp32 division)
 *               q      = E2M1_rn_satfinite(v / value(s_code))   (IEEE fp32 division)
 *             tensor-level scale 1;
 *   FP8_B128  per block of 128 consecutive elements of a row:
 *               s = amax / 448 (fp32, IEEE division),  q = E4M3_rn_satfinite(v / s)
 * with q a zero of v's sign when the scale is 0.  This call applies the rule to
 * x [T][d] (bf16) in token order:
 *   NVFP4     codes uint8 [T][d/2] (element 2i in the low nibble of byte i),
 *             scales uint8 [T][d/16] (E4M3 codes)
 *   FP8_B128  codes uint8 [T][d] (E4M3), scales float [T][d/128] (4-byte aligned)
 * Other formats: NVFP4's rule.  Preconditions: 1 <= T <= 2^20, d % 256 == 0.
 * ------------------------------------------------------------------------- */
ftmoe_status ftmoe_quantize_act(const ftmoe_layer_desc* desc, const uint16_t* x, int T, uint8_t* codes,
                                uint8_t* scales, void* stream);

/* ---------------------------------------------------------------------------
 * a2  ftmoe_permute - stable expert-sorted permutation of the P = T*k pairs.
 * The pages do not describe it.  It is what computing each selected expert
 * once over a batch needs (banandre.com, section "Sparsity Is a Lie").
 *   topk_ids        int32 [T][k], every id in [0, E)
 *   expert_offsets  int32 [E+1]: exclusive prefix sum of per-expert counts
 *   sorted_pair     int32 [P]: pair indices p = t*k + r ordered by (expert, p)
 *   pair_pos        int32 [P]: position of pair p in sorted_pair
 * An id outside [0, E) sets FTMOE_ERR_DEVICE_CHECK and is counted as expert E-1.
 * ------------------------------------------------------------------------- */
size_t ftmoe_permute_workspace_size(const ftmoe_layer_desc* desc, int T);
ftmoe_status ftmoe_permute(const ftmoe_layer_desc* desc, const int32_t* topk_ids, int T,
                           int32_t* expert_offsets, int32_t* sorted_pair, int32_t* pair_pos,
                           void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * a3+a4  ftmoe_expert_ffn - grouped SwiGLU FFN of the resident experts.
 * Pages: resident experts are computed on GPU tensor cores from expert slots
 * (zubnet.ai, "FreeToken, Unsloth GGUF ... consumer hardware").
 * For each expert e with slot_of[e] >= 0, over its rows
 * sorted_pair[expert_offsets[e] .. expert_offsets[e+1]):
 *   h = silu(X W_gate^T) * (X W_up^T),   y = h W_down^T
 * where X holds the rows x[p / k] of those pairs.  Experts with slot_of[e] < 0
 * are skipped: that is one side of an exact split.
 *   slot_of   int32 [E]: slot index in `weights`, or -1.  An entry >= weights->C
 *             is a data error: that expert is skipped and the device error word
 *             is set (code 2)
 *   topk_w    NULL: y_or_out is y, fp32 [P][d] in sorted order (row j = pair
 *             sorted_pair[j]); rows of skipped experts are left untouched
 *             otherwise: fused combine.  y_or_out is out fp32 [T][d], and
 *             w[p] * y is ADDED into it (zero it first, or pass a partial to merge)
 * Paths (ftmoe_expert_ffn_path tells which one a call takes):
 *   0  weight-only streaming: no activation quantisation.  For NVFP4 / MXFP4
 *      weights the decoded weights meet x and h rounded to f16 in warp-level
 *      MMAs with fp32 accumulation; BF16 and FP8 weights run on CUDA cores in
 *      fp32.  Small T (decode), and every format the tensor-core path does not
 *      cover.  A call on this path takes at most (T*k/8 + E) * max(d, ffn) <= 2^28
 *      work items (a 16384-token chunk at d 4096, top-6: 5.1e7); larger calls
 *      return FTMOE_ERR_UNSUPPORTED and are split by tokens.
 *   1  NVFP4 weights, T >= FTMOE_PREFILL_MIN_T, d % 256 == 0, ffn % 256 == 0:
 *      tcgen05 block-scaled tensor cores.  The gathered rows of x and h are
 *      quantised to NVFP4 by the rule of ftmoe_quantize_act.  Needs
 *      weights->prepared (FTMOE_ERR_INVALID_ARG without it).  With topk_w the
 *      combine is fused (fp32 atomic adds, so the order of the k adds into
 *      out varies between runs); without it y is written in sorted order.
 *   2  FP8_B128 weights, T >= FTMOE_PREFILL_MIN_T, d % 256 == 0, ffn % 128 == 0,
 *      d and ffn <= 8192: tcgen05 FP8 tensor cores.  x and h are quantised to
 *      E4M3 with one fp32 scale per (row, 128 columns) (rule of
 *      ftmoe_quantize_act); each 128-wide K step's fp32 partial is scaled by the
 *      activation and weight block scales and accumulated in fp32.  Combine as
 *      for path 1.  Reads the canonical arena (no preparation).
 * ------------------------------------------------------------------------- */
#define FTMOE_PREFILL_MIN_T 256
size_t ftmoe_expert_ffn_workspace_size(const ftmoe_layer_desc* desc, int T);
/* Which path ftmoe_expert_ffn takes for this layer and T: 0 = weight-only streaming
 * on CUDA cores (no activation quantisation), 1 = tensor cores with NVFP4
 * activations, 2 = tensor cores with FP8 activations.  -1 = invalid descriptor. */
int ftmoe_expert_ffn_path(const ftmoe_layer_desc* desc, int T);
ftmoe_status ftmoe_expert_ffn(const ftmoe_layer_desc* desc, const ftmoe_weights* weights,
                              const int32_t* slot_of, const uint16_t* x, int T,
                              const int32_t* expert_offsets, const int32_t* sorted_pair,
                              const float* topk_w, float* y_or_out,
                              void* ws, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------------------
 * a5  ftmoe_combine - weighted combine and exact merge.
 * Pages: the partial sums over a split of the selected experts add up exactly
 * once the layer completes (banandre.com, section "The q* Policy").
 *   out_t = partial_b_t + sum_{r: slot_of[ids[t,r]] >= 0} w[t,r] * y[pair_pos[t*k+r]]
 * summed in ascending r, in fp32.
 *   y          fp32 [P][d] sorted rows, or NULL (then out = partial_b, a cast/merge only)
 *   slot_of    int32 [E] or NULL (= every expert resident); this call does not know
 *              the arena, so every entry >= 0 counts as resident
 *   partial_b  fp32 [T][d] or NULL
 *   out_f32    fp32 [T][d] or NULL; out_bf16 bf16 [T][d] or NULL (round to nearest even)
 * ------------------------------------------------------------------------- */
ftmoe_status ftmoe_combine(const ftmoe_layer_desc* desc, int T, const float* y, const int32_t* pair_pos,
                           const float* topk_w, const int32_t* topk_ids, const int32_t* slot_of,
                           const float* partial_b, float* out_f32, uint16_t* out_bf16, void* stream);

/* ---------------------------------------------------------------------------
 * a6  global LRU slot map over (layer, expert) keys, key = layer*E + e.
 * Pages: at decode time one LRU, global over the layers' experts, admits every
 * missed expert (asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU", section
 * "Abandoning fixed offloading in favor of measured bandwidth").  It spans all
 * MoE layers (banandre.com, section "Semantic-Aware Caching").  It starts
 * cold (banandre.com, section "Elastic Memory").
 * Reading:
 *   - Each call makes one access per unique expert of topk_ids, in ascending id order.
 *   - A hit refreshes the key's recency.
 *   - A miss takes the lowest free slot, else evicts the least recently used key
 *     and takes its slot.
 * The handle owns its device state: slot_of [L][E], key per slot, recency list.
 * ------------------------------------------------------------------------- */
typedef struct ftmoe_lru ftmoe_lru;

/* L layers, E experts per layer, C slots.  The state is processed in shared memory,
 * so (L*E + 3*C) * 4 bytes must stay within 200 KiB (else FTMOE_ERR_UNSUPPORTED).
 * Allocates the handle's device state. */
ftmoe_status ftmoe_lru_create(int L, int E, int C, ftmoe_lru** out);
/* Empties the table (cold start).  Asynchronous on stream. */
ftmoe_status ftmoe_lru_reset(ftmoe_lru* lru, void* stream);
/* Synchronises the device, then frees the state. */
ftmoe_status ftmoe_lru_destroy(ftmoe_lru* lru);
/* Device pointer to the handle's slot_of table, int32 [L][E] (-1 = not resident).
 * Row l is the slot_of argument of ftmoe_expert_ffn for layer l. */
const int32_t* ftmoe_lru_slot_of(const ftmoe_lru* lru);
/* Copies the slot_of table into dst (device, int32 [L][E]); asynchronous on stream. */
ftmoe_status ftmoe_lru_copy_slot_of(const ftmoe_lru* lru, int32_t* dst, void* stream);

/* One call: the accesses of (layer, topk_ids [B][k]).  Outputs are per access,
 * in access order.  Size them for min(B*k, E) entries:
 *   hit uint8, slot int32, evicted_key int32 (-1 = none)
 *   counters int64 [2] or NULL: the handle's running totals (accesses, misses) after the call
 * FTMOE_ERR_INVALID_ARG: NULL handle or output, B or k < 1, B*k above 2^31-1, layer
 * outside [0, L).  An id outside [0, E) is skipped and sets the device error word
 * (ftmoe_get_device_error). */
ftmoe_status ftmoe_slot_lru(ftmoe_lru* lru, int layer, const int32_t* topk_ids, int B, int k,
                            uint8_t* hit, int32_t* slot, int32_t* evicted_key, int64_t* counters,
                            void* stream);
/* A whole trace int32 [steps][L][B][k] in one launch, steps outer, layers inner.
 * Outputs hold every access of the trace in order; capacity (host) is their length.
 *   counters int64 [2] or NULL: running totals (accesses, misses); at most `capacity`
 *   accesses are written.  Needing more sets the device error word.
 * FTMOE_ERR_INVALID_ARG as for ftmoe_slot_lru, and for steps < 1, capacity < 0 or
 * steps*L above 2^31-1. */
ftmoe_status ftmoe_slot_lru_replay(ftmoe_lru* lru, const int32_t* trace, int steps, int B, int k,
                                   uint8_t* hit, int32_t* slot, int32_t* evicted_key, int64_t capacity,
                                   int64_t* counters, void* stream);

/* ---------------------------------------------------------------------------
 * The decode-time expert cache around the LRU (the rows after the hot path).
 * Pages: a missed expert is either copied over the host link into the GPU cache
 * or computed where its weights are; for a step with m misses the engine fills
 * q* ~= m * B_P / B_H of them, B_P the measured link (PCIe) bandwidth and B_H the
 * measured host-memory bandwidth, and the two partial sums merge exactly after
 * the layer (banandre.com, "The 284B Model on a 32GB GPU Trick", section "The q*
 * Policy: Math Instead of Guesses").  The host pool is kept in its final layout
 * in pinned memory, and at scheduler safe points the cache is rebuilt under a
 * new VRAM budget without reloading that pool (same page, section "Elastic
 * Memory: The VRAM Budget Is a Suggestion").
 * Reading: both executors of the split are GPU work.  Executor A computes the
 * experts resident in the HBM slot arena; executor B computes the others with
 * their weights streamed straight from the host pool (an ftmoe_weights whose
 * arrays are pinned host memory the device can address, one slot per
 * (layer, expert), slot layer*E + e, passed with prepared = NULL so that the
 * decode path reads it with plain loads).  out = A + B through ftmoe_combine's
 * partial_b.  Executor B is meant for the decode path (ftmoe_expert_ffn_path 0).
 * ------------------------------------------------------------------------- */

/* ftmoe_copy_slots - copy whole slots from one arena to another (or within one).
 * For i < min(*n_pairs, max_pairs) (n_pairs device int32, or NULL = max_pairs):
 * slot pairs[i][0] of src -> slot pairs[i][1] of dst: codes, scales, tensor
 * scales and, when both arenas carry one, the prepared layouts (both or neither
 * must have prepared; FTMOE_ERR_INVALID_ARG otherwise).  Uses:
 *   - fills: src = the host pool (pinned host memory, read over the host link
 *     by the kernel, zero-copy), dst = the HBM arena, pairs = (layer*E + e, slot);
 *   - compaction after ftmoe_lru_resize shrinks: src = dst = the arena, pairs =
 *     the resize's moves (pairs with equal slots are skipped; the destinations
 *     of a shrink are never sources, so the copies do not overlap);
 *   - migration to an arena of another slot count: pairs = the resize's moves.
 * Pairs outside either arena are skipped and set the device error word.  Two
 * pairs must not share a destination.  The arenas have the layer's shape and
 * format. */
ftmoe_status ftmoe_copy_slots(const ftmoe_layer_desc* desc, const ftmoe_weights* src, const ftmoe_weights* dst,
                              const int32_t* pairs, const int32_t* n_pairs, int max_pairs, void* stream);

/* q* of the pages for m misses, q* = m * link_gbs / host_gbs (fp64), and the fill
 * count: q* rounded half up, clamped to [0, m].  -1 for m < 0 or a bandwidth that is
 * not positive and finite.  Host arithmetic only. */
double ftmoe_qstar(int m, double link_gbs, double host_gbs);
int ftmoe_qstar_fill_count(int m, double link_gbs, double host_gbs);

/* ftmoe_miss_split - split the experts of one ftmoe_slot_lru call between the two
 * executors.  Run right after that call, on the same stream, with its topk_ids
 * [B][k] and hit flags.  Reads the handle's slot table as the call left it.
 *   m = the call's misses; n_fill = fill_override if >= 0, else
 *   ftmoe_qstar_fill_count(m, link_gbs, host_gbs); then, over the call's experts in
 *   ascending id (its accesses):
 *     resident after the call (slot >= 0) and a hit   -> A: slot_of_a[e] = slot
 *     resident, a miss, among the first n_fill such  -> A, and fill_now gets
 *                                                       (layer*E + e, slot)
 *     resident, a miss, beyond those                 -> B: slot_of_b[e] = layer*E + e,
 *                                                       and fill_later gets the pair
 *     not resident (its slot went to a later miss of the same call) -> B
 *   slot_of_a, slot_of_b  int32 [E], -1 where the executor skips the expert
 *   fill_now, fill_later  int32 [min(B*k, E)][2] (pool slot, arena slot)
 *   counts                int32 [4]: m, fills now, fills later, experts of B
 * fill_now must land (ftmoe_copy_slots with n_pairs = counts + 1) before A reads
 * the arena; fill_later (n_pairs = counts + 2) writes only slots that A does not
 * read, so it may overlap both executors.  E <= 1024 (else FTMOE_ERR_UNSUPPORTED). */
ftmoe_status ftmoe_miss_split(const ftmoe_lru* lru, int layer, const int32_t* topk_ids, int B, int k,
                              const uint8_t* hit, double link_gbs, double host_gbs, int fill_override,
                              int32_t* slot_of_a, int32_t* slot_of_b, int32_t* fill_now, int32_t* fill_later,
                              int32_t* counts, void* stream);

/* The handle's current slot count. */
int ftmoe_lru_capacity(const ftmoe_lru* lru);

/* ftmoe_lru_resize - rebuild the slot map under a new capacity C_new, at a safe point
 * (no call on the handle in flight).  Reading of the pages' elastic rebuild:
 *   - the C_new most recently used keys stay resident, in the same recency order;
 *     the others are evicted;
 *   - a kept key in a slot below C_new keeps it; kept keys in slots >= C_new, in
 *     ascending slot order, move to the freed slots below C_new in ascending order,
 *     so the occupied slots stay 0 .. used-1 and later misses take the lowest free
 *     slot; growing keeps every key where it is;
 *   - the running totals carry over.
 *   moves    int32 [min(C_old, C_new)][2] or NULL: (old slot, new slot) of every kept
 *            key, in ascending old slot (the pairs for ftmoe_copy_slots)
 *   n_moves  int32 [1] or NULL: the kept keys
 * Allocates the new device state, runs on `stream`, synchronises it, then frees the
 * old state.  FTMOE_ERR_UNSUPPORTED if (L*E + 3*C_new) * 4 bytes exceed 200 KiB. */
ftmoe_status ftmoe_lru_resize(ftmoe_lru* lru, int C_new, int32_t* moves, int32_t* n_moves, void* stream);

/* ftmoe_layers_streamed - L MoE layers whose experts stream from a host pool larger than
 * the device arenas (prefill of a model that does not fit in the GPU's expert budget).
 * Pages: during prefill, full-layer double buffering streams layer l+1's experts while the
 * GPU computes layer l, and turning the second buffer off costs throughput that grows with
 * the prompt length (asapai.co.kr, "Running 753B GLM-5.2 on a single workstation GPU",
 * section "Abandoning fixed offloading in favor of measured bandwidth"; banandre.com, "The
 * 284B Model on a 32GB GPU Trick", section "Semantic-Aware Caching").
 *   pool       the host pool: C >= L*E slots, expert e of layer l in slot l*E + e (pinned
 *              host memory the device can address); it carries a prepared layout when
 *              the arenas do
 *   arenas     n_arenas (1 or 2) device arenas of at least E slots, same format
 *   x          [L] inputs [T][d] bf16 (device); x[l] == NULL for l > 0 takes out_bf16[l-1]
 *   w_router   [L] router weights [E][d];  logit_bias [L] or NULL (entries may be NULL)
 *   out_f32    [L] outputs [T][d] fp32;  out_bf16 [L] or NULL (bf16 outputs)
 *   ws         the layer call's workspace for T (ftmoe_layer_workspace_size)
 * For each layer, one cudaMemcpyAsync per array copies its E experts (a contiguous range
 * of each pool array) into arena l % n_arenas on copy_stream: the canonical arrays and the
 * part of the prepared layout that the call's path reads.  The layer then runs
 * (ftmoe_layer_forward, every expert resident) on compute_stream once its copy has landed.
 * With two arenas the copy of layer l+1 overlaps the compute of layer l; with one it waits
 * for it.  The copy stream first waits for the work already queued on the compute stream,
 * and the compute stream's last layer comes after every copy; the two streams must differ.
 * Asynchronous on both streams. */
ftmoe_status ftmoe_layers_streamed(const ftmoe_layer_desc* desc, int L, const ftmoe_weights* pool,
                                   const ftmoe_weights* arenas, int n_arenas, const uint16_t* const* x,
                                   const uint16_t* const* w_router, const float* const* logit_bias, int T,
                                   float* const* out_f32, uint16_t* const* out_bf16, void* ws, size_t ws_bytes,
                                   void* compute_stream, void* copy_stream);

/* ---------------------------------------------------------------------------
 * Whole layer in one call: route -> permute -> expert FFN -> combine -> bf16.
 * This is the same work as the four calls above, on one workspace.
 *   slot_of    int32 [E] or NULL (every expert resident in slot e); an entry
 *              >= weights->C is skipped in every step and sets the device error word
 *   topk_ids, topk_w  outputs as in ftmoe_route (may be NULL only together)
 *   out_f32    fp32 [T][d] (required);  out_bf16  bf16 [T][d] or NULL
 * Three forms (ftmoe_layer_path tells which one a call takes):
 *   2  one kernel in the slice form: form 1's router and selection, then each
 *      gate/up item also applies its 16 columns of the down projection, and the
 *      CTAs' partial outputs are summed in CTA order at the end.  The sum of form
 *      1 regrouped: equal up to fp32 reassociation, and the same from run to run.
 *   1  one kernel, for T <= 8 with NVFP4 or MXFP4 weights and weights->prepared:
 *      every CTA computes the logits of its share of the experts, one grid-wide
 *      sync, then every CTA selects the top-k and sorts the pairs itself and
 *      streams its share of the selected experts.  The combine is a merge in
 *      ascending rank, as ftmoe_combine computes it, so the results equal the
 *      separate calls' bit for bit.
 *   0  the separate steps on one stream (the expert FFN with fused combine on
 *      the decode path, the combine call otherwise), with the expert FFN's size
 *      limit on its path 0.
 * ------------------------------------------------------------------------- */
size_t ftmoe_layer_workspace_size(const ftmoe_layer_desc* desc, int T);
/* Which form ftmoe_layer_forward takes for these weights and T: 0 = separate steps,
 * 1 = one kernel (T <= 8), 2 = one kernel in the slice form (d <= 2048 and T = 1, or
 * T <= 8 with NVFP4 weights: each
 * gate/up item also applies its 16 columns of the down projection, and the CTAs' partial
 * outputs are summed in a fixed order; the combine's sum regrouped, fp32 reassociation
 * only), -1 = invalid descriptor or weights. */
int ftmoe_layer_path(const ftmoe_layer_desc* desc, const ftmoe_weights* weights, int T);
ftmoe_status ftmoe_layer_forward(const ftmoe_layer_desc* desc, const ftmoe_weights* weights,
                                 const int32_t* slot_of, const uint16_t* x, const uint16_t* w_router,
                                 const float* logit_bias, int T, int32_t* topk_ids, float* topk_w,
                                 float* out_f32, uint16_t* out_bf16, void* ws, size_t ws_bytes,
                                 void* stream);

/* ftmoe_layer_forward_host - the layer call from and to host memory, for callers whose
 * activations live on the host.  On `stream`: x_host [T][d] bf16 (host, pinned for an
 * asynchronous copy) is copied into the workspace, ftmoe_layer_forward runs on it, and
 * the bf16 output is copied back to out_host [T][d] (host).  topk_ids / topk_w and
 * out_f32 stay on the device as in ftmoe_layer_forward (out_f32 required).  The
 * workspace (ftmoe_layer_host_workspace_size) is the layer call's plus staging for x
 * and the bf16 output.  Asynchronous: out_host is valid once the stream reaches the
 * end of the call. */
size_t ftmoe_layer_host_workspace_size(const ftmoe_layer_desc* desc, int T);
ftmoe_status ftmoe_layer_forward_host(const ftmoe_layer_desc* desc, const ftmoe_weights* weights,
                                      const int32_t* slot_of, const uint16_t* x_host, const uint16_t* w_router,
                                      const float* logit_bias, int T, int32_t* topk_ids, float* topk_w,
                                      float* out_f32, uint16_t* out_host, void* ws, size_t ws_bytes, void* stream);

/* ftmoe_layer_graph - one ftmoe_layer_forward_host call recorded once as a CUDA graph and
 * replayed: a decode step of one token issues a copy in, one kernel and a copy out, and a
 * replay costs the host one graph launch instead of three stream operations and the checks
 * around them.
 *   ftmoe_layer_graph_create takes the arguments of ftmoe_layer_forward_host, checks them the
 *   same way, and records the call by stream capture on `stream` (a stream created by the
 *   caller: the legacy default stream cannot be captured; NULL is FTMOE_ERR_INVALID_ARG, as is
 *   a stream already being captured).  Nothing runs at creation.  The pointers are bound into
 *   the graph: every replay copies from x_host and writes out_host, topk_ids, topk_w and
 *   out_f32 as one ftmoe_layer_forward_host call with those arguments would, so the caller
 *   keeps every buffer alive and refills x_host (pinned) between replays; a replay reads the
 *   weights, router and slot table at their bound addresses as they are when it runs.
 *   The caller owns *out; on failure *out is NULL and the stream is no longer capturing.
 *   ftmoe_layer_graph_launch replays on `stream` (any stream of the graph's device; NULL =
 *   the legacy default stream).  Replays on one workspace must not overlap (the rule of the
 *   layer call), so replays of one graph on two streams need an order between them.
 *   ftmoe_layer_graph_destroy frees the graph (NULL is a no-op); replays already issued
 *   still complete.
 * Results equal those of ftmoe_layer_forward_host with the same arguments. */
typedef struct ftmoe_layer_graph ftmoe_layer_graph;
ftmoe_status ftmoe_layer_graph_create(const ftmoe_layer_desc* desc, const ftmoe_weights* weights,
                                      const int32_t* slot_of, const uint16_t* x_host, const uint16_t* w_router,
                                      const float* logit_bias, int T, int32_t* topk_ids, float* topk_w,
                                      float* out_f32, uint16_t* out_host, void* ws, size_t ws_bytes, void* stream,
                                      ftmoe_layer_graph** out);
ftmoe_status ftmoe_layer_graph_launch(ftmoe_layer_graph* graph, void* stream);
ftmoe_status ftmoe_layer_graph_destroy(ftmoe_layer_graph* graph);

/* ---------------------------------------------------------------------------
 * Helpers
 * ------------------------------------------------------------------------- */
const char* ftmoe_status_string(ftmoe_status s);
/* Reads and clears the device error word (synchronises `stream`).
 * *code = 0 if no device-side check failed since the last read. */
ftmoe_status ftmoe_get_device_error(int* code, void* stream);
/* Sets the time after which every bounded device wait of the library gives up (grid and
 * cluster-partial counters, shared-memory barriers, readiness counts): ns, or 0 for the default
 * 2 s.  A wait that gives up sets the device error word (codes 6 and 10 are timeouts) and the
 * kernel winds down without trapping; after one, zero the workspace's first
 * FTMOE_WS_ZERO_BYTES bytes before its next use.  Synchronous; applies to later launches on
 * the current device.  For tests and diagnostics that make a wait run out. */
ftmoe_status ftmoe_set_wait_limit(unsigned long long ns);
/* Library version, e.g. 100 = 0.1.0. */
int ftmoe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* FTMOE_H */
