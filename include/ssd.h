/*
 * ssd.h -- C ABI of the GB300 selective-SSM (Mamba2 SSD) serving library.
 *
 * Three calls make up the serving hot path of a Mamba2 layer's state-space
 * part:
 *
 *   ssd_chunk_metadata  host:   varlen chunk metadata and slot routing
 *   ssd_prefill_varlen  device: chunked SSD prefill scan over packed sequences
 *   ssm_decode_update   device: single/speculative-token decode state update
 *
 * Next to them: the depthwise causal conv1d that produces x, B and C
 * (ssd_conv1d_varlen / ssd_conv1d_update) and the Mamba1 selective scan with
 * per-channel states (mamba1_scan_varlen / mamba1_state_update).
 *
 * The recurrence (per head h, group g = h / (nheads / ngroups)):
 *   delta_t = clamp(softplus(dt[t,h] + dt_bias[h]), dt_min, dt_max)
 *   s_t     = exp(delta_t * A[h]) * s_{t-1} + delta_t * x[t,h,:] (outer) B[t,g,:]
 *   y[t,h]  = s_t . C[t,g,:] + D[h] * x[t,h,:]
 * with s a [headdim, dstate] fp32 state.  This is the selective SSM (S6)
 * whose Delta, B and C depend on the input, as summarised on
 * "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링", section
 * "논문 핵심 내용"; the argument set (dt_bias, dt_softplus, dt_limit, D,
 * grouped B/C, state dtype) is that of the varlen chunk-scan call on
 * "[vllm] vLLM Mamba2 SSD 커널 웜업", section "mamba_mixer2.py 변경 사항 (핵심)".
 *
 * Conventions shared by every call
 *   - All tensors are dense and row-major (last index fastest).
 *   - "device" pointers are CUDA global memory of the current device;
 *     "host" pointers are ordinary CPU memory.  The caller owns every buffer.
 *   - Device calls are asynchronous on the given stream.  They launch CUDA
 *     kernels and return; they never synchronise, never allocate and keep no
 *     state between calls.
 *   - Host-side argument checks return a status synchronously and launch
 *     nothing.  Problems only visible on the device (a slot id outside
 *     [0, num_slots), metadata that contradicts cu_seqlens) set bits in the
 *     optional device word *err_word (atomic OR; the caller zeroes it and
 *     reads it after synchronising); the offending access is skipped.
 *   - A slot id equal to null_block_id is never read or written, even when
 *     null_block_id is itself a valid index such as 0.
 *   - State slots of different sequences / requests must not alias.  Within
 *     one sequence the initial-state slot may equal a chunk's output slot; the
 *     initial state is read before any state of that sequence is written.
 */
#ifndef SSD_GB300_SSD_H
#define SSD_GB300_SSD_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SSD_API __attribute__((visibility("default")))
#else
#define SSD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t (the same type); NULL is the legacy default stream. */
typedef struct CUstream_st *ssd_stream_t;

typedef enum {
    SSD_OK = 0,
    SSD_ERR_INVALID_ARG = 1, /* a size, pointer, alignment or index argument is invalid */
    SSD_ERR_UNSUPPORTED = 2, /* valid request this build does not implement (e.g. a shape no kernel takes) */
    SSD_ERR_WORKSPACE = 3,   /* workspace (or max_chunks) too small */
    SSD_ERR_CUDA = 4         /* a CUDA runtime call or kernel launch failed */
} ssd_status_t;

/* element type of x, dt, B, C and y; A, D, dt_bias and the state are fp32 */
typedef enum { SSD_F32 = 0, SSD_BF16 = 1 } ssd_dtype_t;

/* bits OR-ed into *err_word by the kernels */
#define SSD_DEVERR_SLOT 0x1u     /* a slot id not null and outside [0, num_slots) */
#define SSD_DEVERR_METADATA 0x2u /* chunk metadata inconsistent with cu_seqlens */
#define SSD_DEVERR_COLUMN 0x4u   /* num_accepted_tokens outside [0, state_indices_cols) */
#define SSD_DEVERR_TIMEOUT 0x8u  /* a bounded device-side wait gave up */
#define SSD_DEVERR_INTERNAL 0x10u /* launch configuration not as the kernel requires (bug) */

/* Human-readable name of a status code (static string). */
SSD_API const char *ssd_status_string(ssd_status_t status);

/* ABI version of this header; bumped on any incompatible change. */
#define SSD_ABI_VERSION 2
SSD_API int32_t ssd_abi_version(void);

/* ------------------------------------------------------------------------ *
 * Chunk metadata (host)
 *
 * Follows "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링", section
 * "청크 메타데이터 계산": every chunk holds tokens of a single sequence, and a
 * chunk ends at every absolute multiple of chunk_size so the state can be
 * stored every chunk_size tokens (prefix caching).  A sequence whose
 * num_computed_tokens is not a multiple of chunk_size first closes the
 * unaligned remainder of its previous chunk, then continues with full chunks
 * and a partial tail.  Slot routing follows "MetadataBuilder 초기화"
 * ("all" cache mode keeps one state per block; the default mode keeps one per
 * request).
 * ------------------------------------------------------------------------ */

/* Upper bound on the number of chunks: min(T, 2*S + ceil(T/chunk_size)).
 * Returns -1 for invalid arguments. */
SSD_API int32_t ssd_max_chunks(int32_t num_seqs, int32_t total_tokens, int32_t chunk_size);

/*
 * All pointers are HOST memory.  Inputs:
 *   cu_seqlens          [S+1]  cu_seqlens[0] == 0, non-decreasing; sequence r owns
 *                              packed tokens [cu_seqlens[r], cu_seqlens[r+1]).
 *   num_computed_tokens [S]    tokens of r already processed earlier (>= 0), or
 *                              NULL for all zero.  Sets the absolute position of
 *                              r's first new token and so the chunk alignment.
 *   has_initial_states  [S]    nonzero: r resumes from a stored state; NULL = none.
 *   block_table         [S, block_table_stride] "all" mode: slot of block j of r
 *                              (block j covers absolute positions
 *                              [j*chunk_size, (j+1)*chunk_size)); NULL otherwise.
 *                              block_table_cols = valid columns per row.
 *   state_indices       [S]    default mode (block_table == NULL): r's single slot;
 *                              may be NULL.
 *   null_block_id              slot id meaning "no slot".
 * Outputs (capacity max_chunks, which must be >= the number of chunks K):
 *   cu_chunk_seqlens    [K+1]  chunk k owns tokens [cu_chunk_seqlens[k], cu_chunk_seqlens[k+1]).
 *   seq_idx             [K]    sequence of chunk k.
 *   last_chunk_indices  [S]    (number of chunks of sequences 0..r) - 1: r's last
 *                              chunk when r has new tokens; equal to r-1's entry
 *                              (or -1) when it has none.
 *   chunk_block_col     [K]    absolute position of chunk k's last token / chunk_size
 *                              (may be NULL).
 *   init_slot           [S]    slot r's initial state is read from, or null_block_id
 *                              (may be NULL).  "all" mode: block_table[r,
 *                              (num_computed-1)/chunk_size]; default mode:
 *                              state_indices[r].  Only when has_initial_states[r].
 *   chunk_slot          [K]    slot chunk k's end state is written to, or
 *                              null_block_id (may be NULL).  "all" mode:
 *                              block_table[seq, chunk_block_col]; default mode:
 *                              state_indices[seq] for the sequence's last chunk.
 *   seq_order           [S]    sequences by decreasing number of new tokens (ties in
 *                              index order), or NULL; pass it as ssd_prefill_args.seq_order
 *                              so the longest sequences start first.
 *   num_chunks_out             K.
 * Errors: SSD_ERR_INVALID_ARG for bad sizes, a decreasing cu_seqlens, negative
 * num_computed_tokens, has_initial_states with num_computed_tokens == 0 in
 * "all" mode, or a block column >= block_table_cols; SSD_ERR_WORKSPACE when
 * max_chunks is too small.  Outputs are unspecified after an error.
 */
SSD_API ssd_status_t ssd_chunk_metadata(int32_t num_seqs, int32_t chunk_size, const int32_t *cu_seqlens,
                                const int32_t *num_computed_tokens,
                                const uint8_t *has_initial_states, const int32_t *block_table,
                                int64_t block_table_stride, int32_t block_table_cols,
                                const int32_t *state_indices, int32_t null_block_id,
                                int32_t max_chunks, int32_t *cu_chunk_seqlens, int32_t *seq_idx,
                                int32_t *last_chunk_indices, int32_t *chunk_block_col,
                                int32_t *init_slot, int32_t *chunk_slot, int32_t *seq_order,
                                int32_t *num_chunks_out);

/* ------------------------------------------------------------------------ *
 * Varlen SSD prefill (device)
 *
 * The chunked scan of "[vllm] vLLM Mamba2 SSD 커널 웜업", section
 * "mamba_mixer2.py 변경 사항 (핵심)" (mamba_chunk_scan_combined_varlen with
 * cu_seqlens, cu_chunk_seqlens, last_chunk_indices, seq_idx, optional initial
 * states, dt_softplus, dt_limit, fp32 state), run for every packed sequence,
 * storing the state at the end of every chunk (prefix caching, "청크 기반
 * 프리픽스 캐싱" of the Mamba (SSM) page).
 * ------------------------------------------------------------------------ */
typedef struct ssd_prefill_args {
    int32_t total_tokens; /* T = cu_seqlens[S] */
    int32_t num_seqs;     /* S */
    int32_t num_chunks;   /* K = cu_chunk_seqlens entries - 1 */
    int32_t nheads;       /* H */
    int32_t headdim;      /* P */
    int32_t dstate;       /* N */
    int32_t ngroups;      /* G, divides H */
    int32_t chunk_size;   /* Q (informational; the chunks come from cu_chunk_seqlens) */
    int32_t dtype;        /* ssd_dtype_t of x, dt, B, C and y */
    int32_t dt_softplus;  /* nonzero: delta = softplus(dt + dt_bias) before the clamp */
    float dt_min, dt_max; /* dt_limit clamp; (0, +inf) leaves softplus output as is */
    int32_t num_slots;    /* rows of state_cache */
    int32_t null_block_id;
    /* device pointers */
    const void *x;       /* [T, H, P]  dtype, 16-byte aligned */
    const void *dt;      /* [T, H]     dtype */
    const void *B;       /* [T, G, N]  dtype, 16-byte aligned */
    const void *C;       /* [T, G, N]  dtype, 16-byte aligned */
    const void *z;       /* [T, H, P] dtype, 16-byte aligned, or NULL: output gate, y is replaced by
                            y * silu(z) = y * z / (1 + exp(-z)) (the z argument of the chunk-scan
                            call in "mamba_mixer2.py 변경 사항 (핵심)"; NULL there) */
    const float *A;      /* [H] (negative for a decaying state) */
    const float *D;      /* [H] or NULL (no skip term) */
    const float *dt_bias; /* [H] or NULL (zero) */
    const int32_t *cu_seqlens;         /* [S+1] */
    const int32_t *cu_chunk_seqlens;   /* [K+1] */
    const int32_t *seq_idx;            /* [K] */
    const int32_t *last_chunk_indices; /* [S] */
    const int32_t *init_slot;  /* [S] or NULL (no initial states) */
    const int32_t *chunk_slot; /* [K] or NULL (no state output) */
    float *state_cache;        /* [num_slots, H, P, N] fp32, 16-byte aligned; may be NULL
                                  when init_slot and chunk_slot are both NULL */
    void *y;                   /* [T, H, P] dtype, 16-byte aligned, written for every token */
    uint32_t *err_word;        /* device word or NULL */
    const int32_t *seq_order;  /* [S] device, a permutation of 0..S-1 giving the order in which
                                  sequences are started (longest first balances the GPU), or
                                  NULL for index order; results do not depend on it.  An entry
                                  outside [0, S) or repeated sets SSD_DEVERR_METADATA (a repeated
                                  entry leaves the y of the sequence it displaced unwritten) */
    int64_t wait_limit_cycles; /* watchdog of the tensor-core kernel: SM clock cycles any of its
                                  device-side waits (for a copy, a product or another warp) may
                                  take before the CTA sets SSD_DEVERR_TIMEOUT, lets its own copies
                                  and products finish, frees its tensor memory and exits; 0 selects
                                  the default of 2e9 (about a second).  The CUDA-core kernels have
                                  no such waits and ignore it. */
} ssd_prefill_args;

/* Bytes of device workspace ssd_prefill_varlen needs for these arguments
 * (sizes only are read) on the current device.  0 on invalid sizes.  With
 * up256 rounding up to a multiple of 256: bf16 with headdim 64 and dstate 128
 * (the tensor-core kernel) needs the fp16 copies of B and C and, per head and
 * token, delta and its in-block cumsum: 2*up256(2*T*G*N) + 2*up256(4*H*T)
 * bytes.  When S*H is below half the device's SM count, each sequence is cut
 * into k segments of whole 128-token blocks (k = min(SMs / (S*H), T / S / 256,
 * 8), at least 1) that separate CTAs run, and k > 1 adds
 * up256(4*S*(k-1)*H*P*N) + up256(4*S*(k-1)*H) bytes for the state and decay
 * at the end of each segment but the last.  Every
 * other case (the CUDA-core path) needs up256(4*H*T) + up256(8*H*T) +
 * 2*up256(4*K*H*P*N) for delta, the fp64 cumsum, the chunk states and the
 * states entering each chunk. */
SSD_API size_t ssd_prefill_workspace_size(const ssd_prefill_args *args);

/* Number of CUDA kernels one ssd_prefill_varlen call with these arguments
 * launches on the current device (0 for an empty call, -1 on invalid sizes):
 * 2 for the tensor-core path (3 when it cuts sequences into segments), 4 for
 * the CUDA-core path.  Host only. */
SSD_API int32_t ssd_prefill_kernel_count(const ssd_prefill_args *args);

/*
 * Runs the prefill.  workspace: device memory of at least
 * ssd_prefill_workspace_size(args) bytes, 256-byte aligned, caller-owned,
 * no initial contents required, not shared with a concurrent call.
 * Preconditions checked on the host: sizes > 0 (T, K may be 0: nothing
 * happens), H % G == 0, headdim <= 256, dstate <= 256, the pointers required
 * by the sizes are non-NULL, the alignments above.  Returns SSD_ERR_CUDA if a
 * launch fails.
 */
SSD_API ssd_status_t ssd_prefill_varlen(const ssd_prefill_args *args, void *workspace,
                                size_t workspace_bytes, ssd_stream_t stream);

/*
 * ssd_prefill_varlen_marked -- ssd_prefill_varlen that also records the
 * caller's CUDA event `event_before_fused` (a cudaEvent_t, or NULL) on
 * `stream` right before the call's main kernel: on the tensor-core path after
 * the prep kernel (and the segment pass, when it runs), so that the caller's
 * own events before the call, at this mark and after the call time the
 * preparation and the fused kernel apart; on the CUDA-core path before its
 * first kernel.  Results, checks and errors are those of ssd_prefill_varlen;
 * a failed record returns SSD_ERR_CUDA.
 */
SSD_API ssd_status_t ssd_prefill_varlen_marked(const ssd_prefill_args *args, void *workspace,
                                               size_t workspace_bytes, ssd_stream_t stream,
                                               void *event_before_fused);

/*
 * ssd_prefill_varlen_noalloc -- the prefill for callers that cannot allocate.
 *
 * The pages have no counterpart to this call.  It exists for callers that
 * cannot give the library device memory at call time: a serving engine that
 * reserved all free device memory up front (for its state cache) and hands
 * none out afterwards, or a host that only has this C ABI and no device
 * allocator.  It runs the CUDA-core prefill (the kernels that need scratch
 * memory; for every dtype and shape, including those ssd_prefill_varlen would
 * send to the tensor-core kernel) with its scratch in one file-scope device
 * array of SSD_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds
 * until the process exits.  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Arguments, results and host checks are those of ssd_prefill_varlen, minus
 * the workspace.  The call needs up256(4*H*T) + up256(8*H*T) +
 * 2*up256(4*K*H*P*N) bytes of scratch (up256 rounds up to a multiple of 256;
 * e.g. about 4.3 MB for one 2048-token chunk with H=48, P=64, N=128) and
 * returns SSD_ERR_WORKSPACE when that exceeds SSD_NOALLOC_SCRATCH_BYTES;
 * SSD_ERR_UNSUPPORTED for shapes the CUDA-core path does not take.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it with the context it belongs to; make that
 * first call before any stream capture.  After a device reset the next call
 * finds a new context and looks the address up again (again before any
 * capture).  All calls share the one array, and each call leaves its scratch
 * contents behind; nothing in it needs to start at zero, because with
 * metadata from ssd_chunk_metadata every value a call reads was written
 * earlier in the same call.  Calls whose kernels
 * overlap on the GPU (different streams, or different host threads without
 * ordering) race on the array.
 */
#define SSD_NOALLOC_SCRATCH_BYTES (64u << 20)
SSD_API ssd_status_t ssd_prefill_varlen_noalloc(const ssd_prefill_args *args, ssd_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Decode state update (device)
 *
 * "decode는 순차적 갱신" (decode is a sequential update, "왜 이 설계인가"
 * item 2 of the Mamba (SSM) page), with the state-index table of
 * "MetadataBuilder 초기화" ([batch, 1 + num_spec] or [batch, max_blocks]),
 * the CUDA-graph padding of "CUDA Graph 지원" (padded rows hold
 * NULL_BLOCK_ID and are skipped) and the speculative-decode checkpoint of
 * "왜 이 설계인가" item 4 (num_accepted_tokens picks the state to resume from).
 * ------------------------------------------------------------------------ */
typedef struct ssm_decode_args {
    int32_t batch;          /* R, rows of state_indices (live + padding) */
    int32_t tokens_per_req; /* 1 + num_speculative_tokens */
    int32_t nheads, headdim, dstate, ngroups;
    int32_t dtype;          /* ssd_dtype_t of x, dt, B, C and y */
    int32_t dt_softplus;
    float dt_min, dt_max;
    int32_t num_slots;
    int32_t null_block_id;
    int32_t state_indices_cols; /* columns of a state_indices row, >= tokens_per_req */
    const void *x;  /* [R * tokens_per_req, H, P]; token k of request r is row r*tpr + k */
    const void *dt; /* [R * tokens_per_req, H] */
    const void *B;  /* [R * tokens_per_req, G, N] */
    const void *C;  /* [R * tokens_per_req, G, N] */
    const void *z;  /* [R * tokens_per_req, H, P] or NULL: output gate, y * silu(z) as in prefill */
    const float *A, *D, *dt_bias;      /* [H]; D and dt_bias may be NULL */
    float *state_cache;                /* [num_slots, H, P, N] fp32, updated in place */
    const int32_t *state_indices;      /* [R, state_indices_cols] */
    const int32_t *num_accepted_tokens; /* [R] or NULL (all 0): request r resumes from the
                                          state in column num_accepted_tokens[r] */
    void *y;                 /* [R * tokens_per_req, H, P]; rows of skipped requests untouched */
    uint32_t *err_word;      /* device word or NULL */
} ssm_decode_args;

/*
 * Request r with read slot rs = state_indices[r, num_accepted_tokens[r]]:
 * if rs == null_block_id the request is padding and nothing of it is read or
 * written.  Otherwise its state is read from rs, the tokens_per_req tokens are
 * applied in order, y is written for each, and the state after token k is
 * stored to state_indices[r, k] unless that id is null.  The read happens
 * before any write (the read slot may be one of the write slots).
 * Host checks as for prefill, plus tokens_per_req >= 1,
 * state_indices_cols >= tokens_per_req.
 */
SSD_API ssd_status_t ssm_decode_update(const ssm_decode_args *args, ssd_stream_t stream);

/* ------------------------------------------------------------------------ *
 * One step of a mixed batch (device)
 *
 * A scheduled batch holds prefill requests and decode requests, each part
 * with its own metadata and state indices ("BaseMambaAttentionMetadata" on
 * the Mamba (SSM) page: num_prefills / num_decodes, state_indices_tensor_p /
 * _d; "왜 이 설계인가" item 2: the two parts go to different kernels).
 * ------------------------------------------------------------------------ */

/*
 * ssd_mixed_step -- the prefill part and the decode part of one step, issued
 * together.  The result is that of ssd_prefill_varlen(prefill, workspace,
 * workspace_bytes, stream) followed by ssm_decode_update(decode, stream),
 * provided the two parts touch disjoint memory: no state slot that one part
 * reads or writes is written by the other, and their outputs do not overlap
 * (err_word may be the same word).  Either part may be empty
 * (total_tokens == 0 or batch == 0); then this is the other call alone.
 *
 * How it runs: the prefill on a library-owned stream of the device's greatest
 * priority, the decode on one of its least, both forked from `stream` and
 * joined back into it by events, so that work queued on `stream` later waits
 * for both.  On the tensor-core path the decode starts once the prefill's
 * prep kernel is done, so the two bandwidth-bound kernels do not share HBM;
 * it then gets the SMs that the fused prefill kernel leaves idle (a prefill
 * CTA needs a whole SM, and pending prefill CTAs, at the greater priority,
 * take every SM that frees up first), chiefly beside the prefill's last,
 * partial wave.  On the CUDA-core path the decode starts at once.
 *
 * Host checks are those of the two calls, all made before anything is
 * queued.  The streams and events are made on the first call in each context
 * (make it before any stream capture) and kept until the process exits; a
 * device reset makes the next call create them anew.  After that first call
 * the step can be captured into a CUDA graph on `stream`: the fork onto the
 * library's streams and the join back are captured with it.  Calls from several host
 * threads queue their work one call at a time.  Returns SSD_ERR_CUDA if a
 * launch or a stream or event operation fails.
 */
SSD_API ssd_status_t ssd_mixed_step(const ssd_prefill_args *prefill, void *workspace, size_t workspace_bytes,
                                    const ssm_decode_args *decode, ssd_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Depthwise causal conv1d before the SSM (device)
 *
 * The step that produces x, B and C: "get hidden_states, B and C after
 * depthwise convolution" in the MambaMixer2 listing of "[vllm] vLLM Mamba2 SSD
 * 커널 웜업", with a conv state per cache block of shape [state_len, conv_dim]
 * ("vLLM v0.20.0 하이브리드 SSM 모델을 위한 분산 서빙 추가", "전체 흐름": a
 * [num_blocks, 3, 3072] conv tensor next to the [num_blocks, 48, 64, 128]
 * SSM tensor).  For channel c and token t of a sequence,
 *   out[t, c] = act(bias[c] + sum_{k<W} weight[c, k] * in[t - (W-1) + k, c]),
 * where the W-1 inputs before the sequence's first token come from its conv
 * state (zeros without one) and act is silu or the identity.  The conv state
 * after a token is the last W-1 inputs up to and including it (exact copies,
 * in the token dtype).
 * ------------------------------------------------------------------------ */
typedef struct ssd_conv1d_args {
    int32_t total_tokens;  /* T */
    int32_t num_seqs;      /* S (for ssd_conv1d_update: requests R, each tokens_per_req tokens) */
    int32_t num_chunks;    /* K = cu_chunk_seqlens entries - 1, or 0 when chunk_slot is NULL */
    int32_t tokens_per_req; /* ssd_conv1d_update only: tokens of each request (>= 1) */
    int32_t dim_x;         /* channels [0, dim_x) go to x_out */
    int32_t dim_bc;        /* channels [dim_x, dim_x + dim_bc) to B_out, the next dim_bc to C_out */
    int32_t width;         /* W, 2..4 taps */
    int32_t dtype;         /* ssd_dtype_t of xbc, the outputs and conv_state */
    int32_t activation;    /* 0: identity, 1: silu */
    int32_t num_slots;     /* rows of conv_state */
    int32_t null_block_id;
    /* device pointers */
    const void *xbc;       /* [T, D] with D = dim_x + 2 dim_bc, 16-byte aligned rows (D % 8 == 0) */
    const float *weight;   /* [D, W], 16-byte aligned */
    const float *bias;     /* [D] or NULL */
    const int32_t *cu_seqlens;        /* [S+1] (ssd_conv1d_varlen) */
    const int32_t *cu_chunk_seqlens;  /* [K+1] or NULL (ssd_conv1d_varlen) */
    const int32_t *last_chunk_indices; /* [S], chunk ranges as for ssd_prefill_varlen, or NULL */
    const int32_t *init_slot;  /* [S] or NULL: conv state each sequence starts from (null id: zeros);
                                  for ssd_conv1d_update the request's slot, read and then overwritten */
    const int32_t *out_slot;   /* [S] or NULL: where the state after each sequence's last token goes */
    const int32_t *chunk_slot; /* [K] or NULL: where the state after each chunk's last token goes */
    void *conv_state;      /* [num_slots, W-1, D] dtype, 16-byte aligned */
    void *x_out;           /* [T, dim_x]  dtype, 16-byte aligned */
    void *B_out;           /* [T, dim_bc] dtype, 16-byte aligned */
    void *C_out;           /* [T, dim_bc] dtype, 16-byte aligned */
    uint32_t *err_word;    /* device word or NULL (SSD_DEVERR_SLOT for an out-of-range slot) */
} ssd_conv1d_args;

/*
 * Prefill: packed sequences, cu_seqlens as for ssd_prefill_varlen (the chunk
 * metadata of ssd_chunk_metadata gives cu_chunk_seqlens, last_chunk_indices
 * and the slots).  Every conv-state read happens before any conv-state write,
 * so a sequence's initial slot may also be one of its output slots.  Host
 * checks: sizes, dim_x and dim_bc multiples of 8, 2 <= W <= 4, pointers and
 * alignments; SSD_ERR_CUDA if a launch fails.  Two kernels (the convolution,
 * then the state stores).
 */
SSD_API ssd_status_t ssd_conv1d_varlen(const ssd_conv1d_args *args, ssd_stream_t stream);

/*
 * Decode: R requests of tokens_per_req tokens each (token k of request r is
 * row r * tokens_per_req + k), the conv state read from init_slot[r] and the
 * state after the last token written back to the same slot.  A request whose
 * slot is null_block_id is CUDA-graph padding ("CUDA Graph 지원" of the Mamba
 * (SSM) page): none of its rows is read or written.  cu_seqlens,
 * cu_chunk_seqlens, last_chunk_indices, out_slot and chunk_slot are ignored.
 */
SSD_API ssd_status_t ssd_conv1d_update(const ssd_conv1d_args *args, ssd_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Mamba1 selective scan (device)
 *
 * The S6 layer of the Mamba paper as "[vLLM] Mamba (SSM): 선형 시간 복잡도
 * 시퀀스 모델링" summarises it in "논문 핵심 내용": Delta, B and C are
 * functions of the token, and every channel d keeps its own state vector
 * s[d, 0..N-1] with its own decay rates A[d, n] (Mamba2 ties the rate to the
 * head).  Per channel d, group g = d / (dim / ngroups):
 *   delta   = clamp(softplus(dt[t,d] + dt_bias[d]), dt_min, dt_max)
 *   s[d,n] <- exp(delta * A[d,n]) * s[d,n] + delta * x[t,d] * B[t,g,n]
 *   y[t,d]  = sum_n C[t,g,n] * s[d,n] + D[d] * x[t,d]   (then y * silu(z[t,d]) if z)
 * Mamba1 has no chunk of its own; prefix caching takes the state out every
 * chunk_size tokens, 2048 by default for Mamba1 ("[vllm] vLLM Mamba2 SSD 커널
 * 웜업", "vllm/config/model.py 변경 사항").  The chunk metadata and slot
 * routing are those of ssd_chunk_metadata, and decode follows the same
 * state-index, padding and speculative-token rules as ssm_decode_update.
 * ------------------------------------------------------------------------ */
typedef struct mamba1_args {
    int32_t total_tokens;   /* T (mamba1_state_update: batch * tokens_per_req) */
    int32_t num_seqs;       /* S (mamba1_state_update: batch R, rows of state_indices) */
    int32_t num_chunks;     /* K (mamba1_scan_varlen) */
    int32_t tokens_per_req; /* mamba1_state_update: 1 + num_speculative_tokens */
    int32_t dim;            /* channels Dc (d_inner), a multiple of 64 */
    int32_t dstate;         /* N, 8 or 16 */
    int32_t ngroups;        /* G; dim / G is a multiple of 64 (Mamba1: G = 1) */
    int32_t dtype;          /* ssd_dtype_t of x, dt, B, C, z and y */
    int32_t dt_softplus;
    float dt_min, dt_max;
    int32_t num_slots;
    int32_t null_block_id;
    int32_t state_indices_cols; /* mamba1_state_update: columns of a state_indices row */
    /* device pointers */
    const void *x;  /* [T, Dc], 16-byte aligned */
    const void *dt; /* [T, Dc], 16-byte aligned */
    const void *B;  /* [T, G, N], 16-byte aligned */
    const void *C;  /* [T, G, N], 16-byte aligned */
    const void *z;  /* [T, Dc] or NULL, 16-byte aligned: output gate */
    const float *A; /* [Dc, N], 16-byte aligned */
    const float *D; /* [Dc] or NULL */
    const float *dt_bias;              /* [Dc] or NULL */
    const int32_t *cu_seqlens;         /* scan: [S+1] */
    const int32_t *cu_chunk_seqlens;   /* scan: [K+1] */
    const int32_t *last_chunk_indices; /* scan: [S] */
    const int32_t *init_slot;          /* scan: [S] or NULL */
    const int32_t *chunk_slot;         /* scan: [K] or NULL */
    const int32_t *state_indices;      /* update: [R, state_indices_cols] */
    const int32_t *num_accepted_tokens; /* update: [R] or NULL */
    float *state_cache;                /* [num_slots, Dc, N] fp32, 16-byte aligned */
    void *y;                           /* [T, Dc], 16-byte aligned */
    uint32_t *err_word;                /* device word or NULL */
} mamba1_args;

/*
 * Varlen prefill over packed sequences: sequence r starts from
 * state_cache[init_slot[r]] (zeros when null or when init_slot is NULL), and
 * the state after the last token of chunk k goes to chunk_slot[k] unless null.
 * All reads of a sequence's initial state happen before its first write.
 * Host checks: sizes, dim % 64 == 0, (dim / ngroups) % 64 == 0, dstate in
 * {8, 16}, pointers and alignments; SSD_ERR_CUDA if the launch fails.  One
 * kernel.
 */
SSD_API ssd_status_t mamba1_scan_varlen(const mamba1_args *args, ssd_stream_t stream);

/*
 * Decode: request r resumes from state_indices[r, num_accepted_tokens[r]]
 * (padding when that id is null: nothing of r is read or written), applies its
 * tokens_per_req tokens in order, writes y for each and stores the state after
 * token k to state_indices[r, k] unless null.  Host checks as for the scan,
 * plus tokens_per_req >= 1 and state_indices_cols >= tokens_per_req.  One kernel.
 */
SSD_API ssd_status_t mamba1_state_update(const mamba1_args *args, ssd_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* SSD_GB300_SSD_H */
