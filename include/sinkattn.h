/*
 * sinkattn.h -- C ABI of libsinkattn.so: causal / sliding-window / varlen
 * attention with one learnable sink logit per query head, forward and
 * backward, on one NVIDIA GB300 (sm_103a).
 *
 * What is computed. Page "GPT-OSS Agentic RL Training: A Practical
 * Retrospective", section "The Role of Attention Sinks": each head has a
 * learnable scalar S_h that acts as a virtual token inside the softmax; section
 * "Implementation in FlashAttention v3": a forward with sinks, plus a backward
 * that also returns dL/dS_h. The pages give no formula; this library takes the
 * plain reading: exp(S_h) joins the softmax denominator and the virtual token
 * has no value vector. For sequence b, query head h, local row i and every key
 * j the mask allows:
 *
 *     s_ij  = scale * q_i . k_j            (k, v of kv head h / (Hq / Hkv))
 *     LSE_i = log(exp(S_h) + sum_j exp(s_ij))        (natural log)
 *     P_ij  = exp(s_ij - LSE_i),   O_i = sum_j P_ij v_j
 *     dS_h  = - sum_{b,i} exp(S_h - LSE_i) * (dO_i . O_i)
 *
 * and dq, dk, dv are the gradients of the same function (dk, dv summed over
 * the query heads that share a kv head).
 *
 * Mask. Key j is visible from row i (both local to their sequence) iff
 * j <= i when causal, and additionally i - j < window when window > 0: a
 * window of W keys is the W most recent keys, the diagonal included.
 * Sequences never see each other.
 *
 * Data layout (all device memory, caller-owned), d = head_dim (64 or 128):
 *   q        bf16 [total, Hq,  d], token row stride q_row_stride elements
 *   k, v     bf16 [total, Hkv, d], token row strides k_row_stride, v_row_stride
 *   o, dout, dq   bf16 [total, Hq, d] contiguous
 *   dk, dv        bf16 [total, Hkv, d] contiguous
 *   lse      fp32 [Hq, total] (head-major)
 *   sinks, dsinks  fp32 [Hq]
 *   cu_seqlens int32 [nseq + 1]: cu[0] = 0, non-decreasing, cu[nseq] = total.
 * Within a token row the heads are contiguous (head stride d) and the d
 * features are contiguous. Row strides must be multiples of 8 elements and
 * every tensor pointer must be 16-byte aligned.
 *
 * Ownership and threading. The library never allocates or frees device
 * memory: the caller passes a workspace of at least the size the matching
 * *_workspace_size() call returns. All work is enqueued on the given stream
 * (a cudaStream_t passed as void*; NULL = legacy default stream) and the call
 * returns without synchronising. Two calls that share a workspace must not
 * overlap on the GPU.
 *
 * Errors. Arguments are checked on the host before anything is launched;
 * a bad argument returns SINKATTN_ERR_INVALID_ARG or SINKATTN_ERR_UNSUPPORTED
 * and launches nothing. cu_seqlens lives on the device and is checked there:
 * a malformed array makes every kernel skip its work and records
 * SINKATTN_ERR_INVALID_ARG in the device error word. Every wait inside a
 * kernel is bounded; a wait that runs out records SINKATTN_ERR_TIMEOUT in the
 * same word and the kernel returns. sinkattn_device_error() reads the word.
 * A failed launch returns SINKATTN_ERR_CUDA. On any error the outputs are
 * undefined. sinkattn_last_error_message() gives detail for the calling
 * host thread.
 */
#ifndef SINKATTN_H_
#define SINKATTN_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SINKATTN_API __attribute__((visibility("default")))
#else
#define SINKATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum sinkattn_status {
  SINKATTN_OK = 0,
  SINKATTN_ERR_INVALID_ARG = 1,
  SINKATTN_ERR_UNSUPPORTED = 2,
  SINKATTN_ERR_CUDA = 3,
  SINKATTN_ERR_WORKSPACE = 4,
  SINKATTN_ERR_TIMEOUT = 5
} sinkattn_status;

/* Forward: O and LSE (section "Implementation in FlashAttention v3", step 1). */
typedef struct sinkattn_fwd_params {
  const void* q;               /* bf16, see layout above                      */
  const void* k;
  const void* v;
  const float* sinks;          /* fp32 [Hq]; NULL = no sink (S_h = -inf)      */
  const int32_t* cu_seqlens;   /* device int32 [nseq + 1]                     */
  void* o;                     /* out: bf16 [total, Hq, d]                    */
  float* lse;                  /* out: fp32 [Hq, total]; may be NULL          */
  void* workspace;             /* >= sinkattn_fwd_workspace_size() bytes       */
  size_t workspace_bytes;
  void* timing_events[2];      /* optional cudaEvent_t pair recorded on the
                                  stream just before and just after the main
                                  attention kernel; NULL entries = none      */
  int64_t q_row_stride;        /* elements between tokens; 0 = Hq * d         */
  int64_t k_row_stride;        /* 0 = Hkv * d                                 */
  int64_t v_row_stride;        /* 0 = Hkv * d                                 */
  int32_t nseq;                /* >= 0                                        */
  int32_t total;               /* tokens = cu_seqlens[nseq] >= 0              */
  int32_t max_seqlen;          /* >= every sequence length (checked on device) */
  int32_t Hq;                  /* query heads, a multiple of Hkv              */
  int32_t Hkv;                 /* key/value heads                             */
  int32_t head_dim;            /* d: 64 or 128 (else SINKATTN_ERR_UNSUPPORTED) */
  int32_t causal;              /* 1 = causal mask, 0 = none                   */
  int32_t window;              /* <= 0: no window; W > 0 needs causal = 1     */
  float softmax_scale;         /* <= 0 selects 1/sqrt(head_dim)               */
  void* bwd_workspace;         /* optional (NULL = none): the workspace the
                                  backward of this same problem will use. The
                                  forward then prepares it: clears the fp32 dq
                                  accumulator in it while it computes (it has
                                  memory bandwidth to spare; the backward's
                                  first pass does not) and builds the
                                  backward's key-tile list beside its own.
                                  That backward, called with
                                  workspace_cleared = 1 and nothing written to
                                  the workspace in between, skips both.
                                  Ignored by the backward, and at head_dim
                                  128 (whose backward has no dq accumulator
                                  and builds its own lists).                 */
  size_t bwd_workspace_bytes;  /* >= sinkattn_bwd_workspace_size() when set    */
} sinkattn_fwd_params;

/* Backward: dq, dk, dv and dL/dS_h (same section, step 2). The forward fields
 * must describe the same problem the forward ran on; o and lse are its
 * outputs. */
typedef struct sinkattn_bwd_params {
  sinkattn_fwd_params fwd;     /* fwd.o, fwd.lse are inputs here (lse required);
                                  fwd.workspace is ignored                    */
  const void* dout;            /* bf16 [total, Hq, d] contiguous: dL/dO        */
  void* dq;                    /* out: bf16 [total, Hq, d]                     */
  void* dk;                    /* out: bf16 [total, Hkv, d]                    */
  void* dv;                    /* out: bf16 [total, Hkv, d]                    */
  float* dsinks;               /* out: fp32 [Hq]; may be NULL; the gradient is
                                  zero when sinks is NULL                     */
  void* workspace;             /* >= sinkattn_bwd_workspace_size() bytes       */
  size_t workspace_bytes;
  void* timing_events[2];      /* optional, around the main backward kernel    */
  int32_t accumulate_dsinks;   /* 0: dsinks = dL/dS_h; nonzero: dsinks +=
                                  dL/dS_h (gradient accumulation over several
                                  calls, e.g. micro-batches or groups of
                                  sequences of one batch)                     */
  int32_t deterministic;       /* 0: dq is summed over key tiles with atomic
                                  adds (fastest; the order of the sum, and so
                                  the last bits of dq, can change from run to
                                  run). Nonzero: dq comes from a second,
                                  query-stationary pass that sums the key
                                  tiles of each query tile in a fixed order,
                                  so every output is bit-identical from run to
                                  run (dk, dv and dsinks always are). At
                                  head_dim 128 the backward always takes dq
                                  from that pass: tensor memory holds its dK
                                  and dV accumulators with no room for dQ.  */
  void* timing_events_dq[2];   /* optional, around the deterministic dq pass
                                  (ignored when deterministic = 0)           */
  int32_t workspace_cleared;   /* nonzero: the forward of this same problem
                                  prepared this workspace (fwd.bwd_workspace:
                                  the dq accumulator cleared, the key-tile
                                  list built) and nothing has written to it
                                  since; the backward skips those steps.
                                  Ignored when deterministic and at head_dim
                                  128.                                       */
} sinkattn_bwd_params;

/* Workspace sizes in bytes for a problem of this shape (0 on bad input).
 * sinkattn_bwd_workspace_size covers either backward mode; the deterministic
 * one needs no fp32 dq accumulator, and sinkattn_bwd_workspace_size_mode gives
 * the size for the chosen mode (deterministic != 0: the smaller one). At
 * head_dim 128 both give the deterministic size. */
SINKATTN_API size_t sinkattn_fwd_workspace_size(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim);
SINKATTN_API size_t sinkattn_bwd_workspace_size(int32_t nseq, int32_t total, int32_t Hq, int32_t Hkv,
                                   int32_t head_dim);
SINKATTN_API size_t sinkattn_bwd_workspace_size_mode(int32_t nseq, int32_t total, int32_t Hq,
                                                     int32_t Hkv, int32_t head_dim,
                                                     int32_t deterministic);

/* Enqueue the forward / backward on `stream`. */
SINKATTN_API sinkattn_status sinkattn_fwd(const sinkattn_fwd_params* params, void* stream);
SINKATTN_API sinkattn_status sinkattn_bwd(const sinkattn_bwd_params* params, void* stream);

/* Backward with no caller workspace, for callers that cannot allocate device
 * memory when they call the library: a host that has already handed the
 * whole device to its own memory pool, or code that runs where an
 * allocation's implicit synchronisation is not allowed. Same parameters,
 * results and errors as sinkattn_bwd; params->workspace and workspace_bytes
 * are ignored. The pages this library follows have no counterpart to this
 * entry point.
 *
 * The scratch memory is one array inside the library of
 * SINKATTN_STATIC_BWD_WORKSPACE_BYTES bytes, held by every GPU that loads the
 * library until the process exits. A problem whose workspace for the chosen
 * mode, sinkattn_bwd_workspace_size_mode(..., params->deterministic), exceeds
 * it returns SINKATTN_ERR_WORKSPACE and launches nothing. The atomic mode needs
 * 256 bytes of fp32 dq accumulator per (token, query head), so it fits up to
 * about 250 000 (token, query head) rows; the deterministic mode needs a few
 * bytes per row and fits far larger problems. The array's device address is looked up on the first call
 * made on each device (with that device current), so make that first call
 * before any stream capture. Every call shares the array and it keeps the
 * last call's contents (nothing in it needs to start at zero); calls that
 * overlap on the GPU, on any stream, race on it. */
#define SINKATTN_STATIC_BWD_WORKSPACE_BYTES ((size_t)64 << 20)
SINKATTN_API sinkattn_status sinkattn_bwd_static_workspace(const sinkattn_bwd_params* params,
                                                           void* stream);

/* Decode: one new query row per sequence against a paged KV cache, the
 * inference side of the same attention (page "GPT-OSS Agentic RL Training: A
 * Practical Retrospective", section "Implementation in FlashAttention v3",
 * step 1: the forward with sinks, which the pages took from an inference
 * engine). Sequence b holds seqlens[b] keys, the new token's included, and its
 * query is the row at the last position: it sees keys j in
 * [max(0, L - window), L) (all L keys when window <= 0), plus the sink of its
 * head, so o and lse equal the last row of sinkattn_fwd over the same keys.
 * The keys are split into up to num_splits ranges processed side by side;
 * the partial results are merged with the sink in a second kernel.
 *
 * Layouts (d = head_dim: 64 or 128):
 *   q            bf16 [nseq, Hq, d] contiguous
 *   k_cache,     bf16 [num_blocks, block_size, Hkv, d] contiguous; logical
 *   v_cache      block i of sequence b is physical block block_table[b][i]
 *   block_table  int32 [nseq, max_blocks_per_seq]; entries for blocks past a
 *                sequence's last key or wholly before its window are ignored,
 *                the others must be in [0, num_blocks)
 *   seqlens      int32 [nseq], 0 <= seqlens[b] <= max_blocks_per_seq * block_size
 *   o            bf16 [nseq, Hq, d] (out)
 *   lse          fp32 [Hq, nseq] natural log (out; may be NULL)
 * block_size must be 16, 32, 64 or 128; Hq / Hkv must be 1, 2, 4, 8 or 16.
 * A sequence with no keys gets o = 0 and lse = S_h (the sink alone). Device
 * pointers must be 16-byte aligned, the caches' too. An out-of-range length
 * or block index found on the device sets the device error word
 * (SINKATTN_ERR_INVALID_ARG) and that sequence's outputs are left unwritten. */
typedef struct sinkattn_decode_params {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_table;
  const int32_t* seqlens;
  const float* sinks;          /* fp32 [Hq]; NULL = no sink                    */
  void* o;
  float* lse;
  void* workspace;             /* >= sinkattn_decode_workspace_size() bytes    */
  size_t workspace_bytes;
  int32_t nseq;                /* 0..65535                                     */
  int32_t num_blocks;          /* > 0 physical blocks in each cache            */
  int32_t block_size;          /* tokens per block                             */
  int32_t max_blocks_per_seq;  /* columns of block_table                       */
  int32_t Hq;
  int32_t Hkv;
  int32_t head_dim;            /* d: 64 or 128                                 */
  int32_t window;              /* <= 0: every key; W > 0: the last W keys      */
  int32_t num_splits;          /* key ranges per sequence, 1..64; 0 = choose    */
  float softmax_scale;         /* <= 0 selects 1/sqrt(head_dim)                */
} sinkattn_decode_params;

/* Workspace bytes for a decode problem (0 on bad input): the split partials,
 * (max, sum) and an unnormalised output row per (sequence, head, split).
 * sinkattn_decode_workspace_size is the head_dim 64 size;
 * sinkattn_decode_workspace_size_d takes the head_dim (64 or 128). */
SINKATTN_API size_t sinkattn_decode_workspace_size(int32_t nseq, int32_t Hq, int32_t num_splits);
SINKATTN_API size_t sinkattn_decode_workspace_size_d(int32_t nseq, int32_t Hq, int32_t num_splits,
                                                     int32_t head_dim);

/* Enqueue the decode on `stream`. num_splits = 0 picks the split count from
 * the shape (nseq, Hkv, max_blocks_per_seq * block_size) and the SM count;
 * size the workspace for 64 splits then (or query it with the chosen count). */
SINKATTN_API sinkattn_status sinkattn_decode(const sinkattn_decode_params* params, void* stream);

/* Decode that agrees bit for bit with the training forward. Same parameters
 * and layouts as sinkattn_decode (num_splits is ignored), and the same
 * result up to rounding; here each query row is computed exactly as
 * sinkattn_fwd computes the row at the last position of the same sequence --
 * the same 128-key tiles from the sequence start, the same online-softmax
 * rescaling rule and the same order of every sum -- so o and lse equal that
 * row of sinkattn_fwd bit for bit when the cache holds the same keys and
 * values (section "Correcting Training-Inference Mismatch via Attention
 * Sinks": the inference engine and the training stack must give the same
 * token probabilities). One work unit per (sequence, kv head) walks the
 * sequence's keys in order, without splitting them, so long sequences take
 * longer than with sinkattn_decode. workspace: at least 256 bytes (a work
 * counter, cleared by the call). Cache slots past a sequence's last key and
 * blocks wholly before its window are not read. Block indices out of range
 * set SINKATTN_ERR_INVALID_ARG in the device error word and read as zeros.
 * At head_dim 128 it is the training forward's head_dim 128 kernel in its
 * decode form. */
SINKATTN_API sinkattn_status sinkattn_decode_exact(const sinkattn_decode_params* params, void* stream);

/* Static description of a status code; never NULL. */
SINKATTN_API const char* sinkattn_status_string(int32_t status);

/* Detail of the last error returned to the calling host thread ("" if none). */
SINKATTN_API const char* sinkattn_last_error_message(void);

/* Synchronises the current device and returns its device error word
 * (SINKATTN_OK if no kernel recorded an error); clears it when reset != 0.
 * Returns SINKATTN_ERR_CUDA if the word cannot be read. */
SINKATTN_API int32_t sinkattn_device_error(int32_t reset);

/* Time limit, in nanoseconds, of every wait inside the library's kernels
 * (an mbarrier phase, a copy landing, a product completing). 0 restores the
 * default of 2 s. It applies to calls enqueued after it, from any thread. A
 * wait that runs out records SINKATTN_ERR_TIMEOUT in the device error word;
 * the kernel then stops its other waits, lets the copies and products it
 * issued finish, frees its tensor memory and returns, so the CUDA context stays
 * usable. No passage of the pages corresponds to this: it is the library's
 * watchdog. */
SINKATTN_API void sinkattn_set_wait_limit_ns(uint64_t ns);

/* Test hook for that watchdog. While on (nonzero), the copy-issuing warp of
 * every pipelined kernel -- the forward, the backward main kernel, the
 * deterministic dq pass and the decode split kernel -- hands out its first
 * work item and then issues no copies, so the warps waiting for them run into
 * the wait limit: the call records SINKATTN_ERR_TIMEOUT, its outputs are
 * undefined, and nothing faults. Applies to calls enqueued after it. Off by
 * default; a test turns it on with a short wait limit and off again. No
 * passage of the pages corresponds to this. */
SINKATTN_API void sinkattn_test_withhold_copies(int32_t on);

/* Number of kernels this library has launched in this process. */
SINKATTN_API uint64_t sinkattn_launch_count(void);

/* sizeof(sinkattn_fwd_params) for which = 0, sizeof(sinkattn_bwd_params) for
 * which = 1, sizeof(sinkattn_decode_params) for which = 2, else 0: lets a
 * binding check its mirror of the structs. */
SINKATTN_API size_t sinkattn_params_size(int32_t which);

#ifdef __cplusplus
}
#endif

#endif /* SINKATTN_H_ */
