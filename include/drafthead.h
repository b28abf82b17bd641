/*
 * drafthead: the reduced-vocabulary draft head of an MTP drafter on one GB300.
 *
 * The drafter's lm_head is restricted to a draft vocabulary: the kept rows of
 * the BF16 target head are gathered (padded to a multiple of 64 rows with
 * copies of the first kept id), quantised to NVFP4 (or per-tensor FP8), and
 * each draft step runs a GEMV of BF16 hidden states against that head with
 * fp32 accumulation, fused with the argmax over kept rows and the map back to
 * target ids. compute_logits scatters the logits into a full-vocabulary fp32
 * row prefilled with -inf.
 *
 * Sources, by page and section:
 *   "q38_draft.py" (Qwen3.8-Flash-Next MTP drafter patch): load_draft_model
 *       (keep mask, dh_idx, pad to N % 64, W[idx] gather, NVFP4 W4A16 head),
 *       get_top_tokens (dh_idx[draft_head(h).argmax(-1)]), compute_logits.
 *   "Qwen3.8-Flash-Next-ABLITERATED - MTP drafter, NVFP4 experts + 98K FP8
 *       head", "How it was built": the NVFP4 recipe (global scale
 *       amax/(6*448), E4M3 block scales per 16, e2m1 round-to-nearest-even)
 *       and the 98,304-row E4M3 per-tensor head.
 *   "FP8 MTP draft stack for vLLM - +6.6% decode on modelopt NVFP4
 *       Qwen3.5-family checkpoints": _fp8_convert_draft_head (amax clamped
 *       at 1e-12, scale = amax/448, clamp, cast) and compute_logits
 *       (new_full(-inf) + index_copy_).
 *
 * Conventions for every entry point:
 *   - Every pointer is a DEVICE pointer unless its name ends in _host.
 *     The caller allocates and owns all memory, workspaces included; the
 *     library never allocates, frees or keeps a pointer after a call returns.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *     enqueue work and return without synchronising, except
 *     draft_head_read_device_error, which synchronises `stream`.
 *   - Arguments are checked on the host before any launch. A failed check
 *     returns a dh_status and launches nothing. Launch failures return
 *     DH_ERR_CUDA. Nothing throws across this interface.
 *   - Faults the host cannot see (a dh_idx entry outside [0, V)) are recorded
 *     in the workspace's device error word; the offending row is skipped.
 *     Read them with draft_head_read_device_error.
 *   - Ids are int32 (V < 2^31); the pages' int64 ids have the same values.
 *   - One call at a time per workspace: two calls in flight on the GPU that
 *     share a workspace race on its argmax slots.
 *   - Draft steps are launched with programmatic stream serialisation: their
 *     kernels start reading the head (q, sf, scale, idx) while the kernel
 *     launched just before them on the same stream may still be running, and
 *     touch h, the workspace and the outputs only after it has completed. So
 *     the kernel immediately preceding a draft step on its stream must not
 *     write that head: after quantising or packing a head on a stream, put any
 *     other operation (an event record, a copy, a memset such as
 *     draft_head_workspace_init, another kernel) between it and the first
 *     draft step, or build the head on another stream and synchronise.
 */
#ifndef DRAFTHEAD_H
#define DRAFTHEAD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DH_ABI_VERSION 1
#define DH_MAX_M 16             /* concurrent drafts per call */
#define DH_WORKSPACE_ALIGN 256  /* required alignment of every workspace */

typedef enum {
    DH_OK = 0,
    DH_ERR_ARG = 1,       /* NULL pointer, unknown format, bad count */
    DH_ERR_SHAPE = 2,     /* shape outside what the kernels support */
    DH_ERR_ALIGN = 3,     /* pointer not aligned as documented */
    DH_ERR_WORKSPACE = 4, /* workspace too small or misaligned */
    DH_ERR_CUDA = 5,      /* a CUDA call or launch failed */
    DH_ERR_TIMEOUT = 6,   /* reserved: a bounded device wait gave up */
    DH_ERR_DEVICE = 7     /* the device error word is set (see below) */
} dh_status;

/* Bits of the device error word. */
#define DH_DEVERR_IDX 1u      /* a dh_idx entry was outside [0, V) */
#define DH_DEVERR_TIMEOUT 2u  /* a bounded device wait gave up (results invalid) */

typedef enum {
    DH_FMT_NVFP4 = 1,
    DH_FMT_FP8 = 2,
    DH_FMT_BF16 = 3,
    DH_FMT_NVFP4_PACKED = 4,
    DH_FMT_FP8_W8A8 = 5
} dh_format;

/* A quantised draft head. Plain descriptor: the library never owns these.
 *   fmt     DH_FMT_NVFP4: q = E2M1 codes [N][K/2], element 2i of a row in the
 *                         low nibble of byte i; sf = E4M3 block scales [N][K/16];
 *                         scale = &g (global scale, 1 float).
 *           DH_FMT_FP8:   q = E4M3 codes [N][K] row-major; sf = NULL;
 *                         scale = &s (per-tensor scale, 1 float).
 *           DH_FMT_BF16:  q = BF16 weights [N][K] row-major; sf = NULL;
 *                         scale = NULL (no scaling).
 *           DH_FMT_NVFP4_PACKED: the NVFP4 head after nvfp4_pack_head: q = the
 *                         tile-major bytes (N * (K/2 + K/16)); sf = NULL;
 *                         scale = &g. Same values, the layout the draft-step
 *                         kernel streams fastest.
 *           DH_FMT_FP8_W8A8: the FP8 head (q, scale as for DH_FMT_FP8) run
 *                         W8A8 ("FP8 MTP draft stack ...",
 *                         _Fp8DraftHeadMethod.apply): each draft step first
 *                         quantises every hidden row to E4M3 with its own
 *                         scale (as fp8_quantize_activations does) and then
 *                         y[m, n] = scale * sx[m] * sum_k q[n, k] * qx[m, k].
 *   V       target vocabulary size (width of the compute_logits rows).
 *   K       hidden size. Supported by the draft-step kernels: 256, 2560
 *           (the pages' drafter hidden size) and 5120.
 *   N       head rows, N % 64 == 0 (the pages pad dh_idx so that N % 64 == 0).
 *   n_kept  rows that are real (1 <= n_kept <= N); rows n_kept..N-1 are the
 *           padding copies of row 0 and take no part in argmax or scatter.
 *   idx     dh_idx [N] int32, target id of each row. May be NULL only for a
 *           BF16 full-vocabulary head (then the row is the id, N == n_kept <= V).
 *   flags   DH_HEAD_IDX_ASCENDING if idx[0..n_kept) is strictly ascending.
 * q and sf must be 16-byte aligned. */
typedef struct dh_head {
    int fmt;
    int V;
    int K;
    int N;
    int n_kept;
    const void *q;
    const uint8_t *sf;
    const float *scale;
    const int32_t *idx;
    unsigned int flags;  /* DH_HEAD_* bits */
} dh_head_t;

/* dh_idx[0..n_kept) is strictly ascending (draft_head_build_index builds it
 * so; keep.nonzero() yields ids in order). Lets get_top_tokens carry target ids
 * in its argmax keys (equal logits still resolve to the lowest row, which then
 * is the lowest id), so the final row -> id lookup drops out. Without it the
 * results are the same. A head without idx (BF16 full vocabulary) counts as
 * ascending. */
#define DH_HEAD_IDX_ASCENDING 1u

/* Build dh_idx on the host ("q38_draft.py", load_draft_model: keep.nonzero(),
 * pad = (-n) % 64 copies of the first kept id). keep_host: V bytes, non-zero =
 * kept. Writes *N ids to idx_host (cap entries available), *n_kept and *N.
 * Errors: DH_ERR_ARG for NULL pointers, V <= 0 or an empty mask (the pages'
 * idx[:1] would be empty); DH_ERR_SHAPE if cap is too small. */
int draft_head_build_index(const uint8_t *keep_host, int V, int32_t *idx_host, int cap,
                           int *n_kept, int *N);

/* Bytes of workspace the quantisers need (a multiple of DH_WORKSPACE_ALIGN). */
size_t draft_head_quantize_workspace_bytes(void);

/* Gather + NVFP4 quantisation of the rows W[idx[n], :], n < N ("Qwen3.8-Flash-
 * Next-ABLITERATED ...", "How it was built"; "q38_draft.py", load_draft_model).
 *   W   BF16 [V][K] row-major target head, 16-byte aligned.
 *   idx int32 [N], entries in [0, V) (out-of-range rows are skipped and set
 *       DH_DEVERR_IDX in the workspace's error word).
 *   q   out [N][K/2] codes; sf out [N][K/16] E4M3 scales; g out: 1 float.
 *   ws  draft_head_quantize_workspace_bytes() bytes, 256-byte aligned.
 * g = max(amax, 1e-12) / 2688 in fp32; per block of 16: s = E4M3_RNE_sat(
 * bamax / fp32(6 g)); codes = E2M1_RNE(clamp(w / fp32(dec(s) g), +-6)) (a
 * zero scale gives signed zeros). K % 16 == 0, N % 64 == 0. Two kernels on
 * `stream`, no host synchronisation. */
int nvfp4_quantize_rows(const void *W, int V, int K, const int32_t *idx, int N,
                        uint8_t *q, uint8_t *sf, float *g, void *ws, size_t ws_bytes,
                        void *stream);

/* Gather + per-tensor FP8 E4M3 quantisation of the rows W[idx[n], :]
 * ("FP8 MTP draft stack ...", _fp8_convert_draft_head): scale =
 * max(amax, 1e-12) / 448 in fp32, q = E4M3_RNE(clamp(w / scale, +-448)),
 * stored row-major [N][K] (the page stores the transpose; same bytes).
 * Arguments as for nvfp4_quantize_rows. */
int fp8_quantize_rows(const void *W, int V, int K, const int32_t *idx, int N,
                      uint8_t *q, float *scale, void *ws, size_t ws_bytes, void *stream);

/* Per-token dynamic FP8 quantisation of hidden states, the activation half of
 * the W8A8 head ("FP8 MTP draft stack ...", _Fp8DraftHeadMethod.apply:
 * scaled_fp8_quant with one scale per token). For each row m < M:
 *   sx[m] = max(max_k |h[m, k]|, 1e-12) / 448   (fp32, IEEE division),
 *   qx[m, k] = E4M3_RNE(clamp(h[m, k] / sx[m], +-448)).
 *   h  BF16 [M][K] row-major, 16-byte aligned; qx out E4M3 codes [M][K],
 *      16-byte aligned; sx out float [M]. M >= 1, K % 16 == 0.
 * One kernel on `stream`; the W8A8 draft step computes the same codes
 * internally, so this call serves callers that want the codes themselves. */
int fp8_quantize_activations(const void *h, int M, int K, uint8_t *qx, float *sx, void *stream);

/* Repack an NVFP4 head into the tile-major layout of DH_FMT_NVFP4_PACKED,
 * the layout Marlin-style GEMV kernels also use instead of the quantiser's
 * row-major one ("q38_draft.py": NVFP4Linear(W, "marlin")). For each tile of
 * 16 rows and each 128-wide k-window w (in that order), `packed` holds a
 * 1,152-byte block: the 16 rows' code bytes 64w..64w+63 (row by row), then
 * 128 bytes of their scales 8w..8w+7: for g < 8 and t < 4, bytes
 * 4 (4 g + t) .. 4 (4 g + t) + 3 hold the scales of blocks 8w + 2t and
 * 8w + 2t + 1 of tile row g, then the same two of tile row g + 8.
 *   q [N][K/2], sf [N][K/16] as written by nvfp4_quantize_rows; packed: device
 *   buffer of N * (K/2 + K/16) bytes. All three 16-byte aligned; N % 16 == 0,
 *   K % 128 == 0. One kernel on `stream`. A pure byte permutation. */
int nvfp4_pack_head(const uint8_t *q, const uint8_t *sf, int N, int K, uint8_t *packed, void *stream);

/* Bytes of workspace the draft-step calls need for up to M_max drafts (a
 * multiple of DH_WORKSPACE_ALIGN). With a head descriptor (hd not NULL,
 * hd->K > 0) the size includes the staging area of draft_head_top_tokens_host
 * for min(M_max, 16) hidden rows of that K; with hd NULL it is the draft-step
 * part alone. */
size_t draft_head_workspace_bytes(const dh_head_t *hd, int M_max);

/* Zero a draft-step workspace (error word, epoch, argmax slots). Call once
 * after allocating it. Draft steps keep it consistent from then on, also
 * after a DH_DEVERR_TIMEOUT: the per-CTA argmax slots alternate between two
 * banks from step to step, the collecting CTA zeroes every slot it read, and
 * a key stored after its collector gave up waiting for it lands in a bank the
 * next step does not read; that step zeroes it before the bank comes round
 * again. */
int draft_head_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* get_top_tokens ("q38_draft.py"): for each draft m < M,
 *   y[m, n] = scale * sum_k w[n, k] * h[m, k]  (fp32 accumulation),
 *   r*      = the lowest row n < n_kept with the largest y[m, n],
 *   ids[m]  = idx[r*]  (or r* when idx is NULL),
 *   top_logit[m] = y[m, r*] if top_logit is not NULL.
 * h: BF16 [M][K] row-major, 16-byte aligned; ids: int32 [M]; 1 <= M <= 16.
 * One kernel launch; capturable in a CUDA graph (no allocation, no sync). */
int draft_head_top_tokens(const dh_head_t *hd, const void *h, int M, int32_t *ids,
                          float *top_logit, void *ws, size_t ws_bytes, void *stream);

/* get_top_tokens for a caller whose hidden states and ids live in host
 * memory (the drafter's loop on the CPU side of a serving process). One call
 * enqueues on `stream`: the copy of h_host (BF16 [M][K] row-major, any
 * alignment) into the staging area at the end of ws, the draft step of
 * draft_head_top_tokens on it, and the copies of the ids (int32 [M]) and,
 * when top_host is not NULL, the top logits (fp32 [M]) back to ids_host /
 * top_host. It returns once they are enqueued; the host results are valid
 * after the stream synchronises. Page-locked host buffers that the device
 * addresses directly (cudaHostAlloc, torch pin_memory(); h 16-byte aligned,
 * ids and top 4-byte aligned) take a path without copy-engine transfers: a
 * one-CTA kernel gathers h into the staging area and the draft step writes
 * the ids (and top logits) into the host buffers. Other host buffers are
 * copied with cudaMemcpyAsync (pageable ones work, but those copies wait on
 * the calling thread, and stream capture refuses them). The caller owns every buffer;
 * ws must be draft_head_workspace_bytes(hd, M_max) bytes with M_max >= M and
 * initialised; calls that overlap on the GPU must not share a workspace.
 * Errors: as draft_head_top_tokens (no alignment rule on the host buffers),
 * DH_ERR_WORKSPACE when ws has no room for M staged rows of this K. */
int draft_head_top_tokens_host(const dh_head_t *hd, const void *h_host, int M, int32_t *ids_host,
                               float *top_host, void *ws, size_t ws_bytes, void *stream);

/* compute_logits ("q38_draft.py" compute_logits; "FP8 MTP draft stack ...",
 * Qwen3_5MTP.compute_logits): out fp32 [M][V] row-major, 16-byte aligned;
 * out[m, :] = -inf, then out[m, idx[n]] = y[m, n] for n < n_kept. idx entries
 * of the kept rows must be distinct. Two kernel launches, both with
 * programmatic stream serialisation: the -inf fill, which writes out only
 * after the kernel before it on the stream has completed, then the GEMV,
 * which writes its logits in place once the fill has completed; capturable
 * in a CUDA graph. */
int draft_head_compute_logits(const dh_head_t *hd, const void *h, int M, float *out,
                              void *ws, size_t ws_bytes, void *stream);

/* One shard of a vocabulary-sharded draft head ("q38_draft.py", install:
 * speculative_config.use_local_argmax_reduction; "FP8 MTP draft stack ...",
 * ParallelLMHead, which splits the head's rows over ranks). A shard is an
 * ordinary head whose dh_idx holds the global target ids of its rows, in
 * strictly ascending order (DH_HEAD_IDX_ASCENDING is required; a BF16 head
 * without idx counts as ascending). Instead of ids, the draft step writes for
 * each draft m < M one int64 key
 *     key[m] = (int64)(((uint64)ord(y*) << 32 | (0xFFFFFFFF - id*)) ^ 2^63)
 * where (y*, id*) is the shard's best (logit, target id): the largest logit,
 * among equal logits the lowest id. ord() maps an fp32 value to uint32
 * preserving order (-0 as +0; every NaN above +inf, as torch.argmax lets NaN
 * win): u | 2^31 for a non-negative value with bits u, ~u for a negative one.
 * The signed maximum of the shards' keys is then the key of the whole head's
 * argmax, so one all-reduce(MAX) of M int64 per step completes the step
 * (draft_head_keys_to_ids decodes it). keys: device int64 [M], 8-byte aligned.
 * Other arguments, workspace and errors as draft_head_top_tokens;
 * DH_ERR_ARG if dh_idx is not flagged ascending. One kernel launch. */
int draft_head_top_keys(const dh_head_t *hd, const void *h, int M, int64_t *keys, void *ws,
                        size_t ws_bytes, void *stream);

/* Decode argmax keys (draft_head_top_keys, combined over shards by a MAX
 * all-reduce) into target ids and, when top_logit is not NULL, the winning
 * logits: id = 0xFFFFFFFF - (key & 0xFFFFFFFF) after undoing the sign flip,
 * logit = the fp32 value whose ord() is the key's high word (NaN for the NaN
 * key). A key of INT64_MIN (no row anywhere) gives id -1. keys: device int64
 * [M]; ids: device int32 [M]; top_logit: device fp32 [M] or NULL; 1 <= M <= 16.
 * One kernel launch on `stream`. */
int draft_head_keys_to_ids(const int64_t *keys, int M, int32_t *ids, float *top_logit, void *stream);

/* NVFP4 W4A16 linear layer of the MTP block ("q38_draft.py", MTP_QUANT_KEYS:
 * fc_embedding, fc_hidden, qkv_proj, o_proj, shared_expert are quantised with
 * the same NVFP4 recipe as the head): for m < M and n < N,
 *   y[m, n] = g * sum_k w'[n, k] * x[m, k]   (fp32 accumulation).
 *   w   an NVFP4 weight in the packed layout: fmt = DH_FMT_NVFP4_PACKED, N
 *       output features (N % 64 == 0), K input features, q = the bytes from
 *       nvfp4_pack_head, scale = &g; V, n_kept, sf, idx and flags are ignored.
 *       Quantise the [N][K] BF16 weight with nvfp4_quantize_rows (idx = 0..N-1).
 *       K in {256, 512, 1024, 2048, 2560, 4096, 5120}.
 *   x   BF16 [M][K] row-major, 16-byte aligned; 1 <= M <= 16.
 *   y   fp32 [M][N] row-major, 16-byte aligned; every entry is written.
 *   ws  a draft-step workspace (draft_head_workspace_bytes bytes, initialised).
 * One kernel launch; capturable in a CUDA graph. */
int nvfp4_linear(const dh_head_t *w, const void *x, int M, float *y, void *ws, size_t ws_bytes,
                 void *stream);

/* get_top_tokens without a caller workspace, for callers that cannot
 * allocate device memory: a plugin hook that is handed only its input and
 * output buffers, or a serving loop that forbids cudaMalloc because it can
 * synchronise the device. The paper has no counterpart of this entry point.
 * Same arguments and results as draft_head_top_tokens, minus the workspace.
 * Its scratch is one fixed array inside the library, laid out as a
 * draft-step workspace (two banks of argmax slots for at most DH_MAX_M = 16
 * drafts, an epoch, an error word; draft_head_workspace_bytes(NULL, 16)
 * bytes); every GPU that loads the library holds it until the process exits.
 * M > 16 returns DH_ERR_SHAPE. The first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture. Each call launches the
 * kernel alone; nothing is allocated. The array is zero at load and stays
 * consistent from step to step, also after a step whose bounded wait ran out
 * (see draft_head_workspace_init). All calls share the one array, so calls
 * that overlap on the GPU (other streams, other threads) race and give wrong
 * ids: serialise them. Device-side faults (a dh_idx entry outside [0, V),
 * which also gives the id -1; a wait that ran out) set bits in the array's
 * error word: read and clear it with draft_head_static_read_device_error. */
int draft_head_top_tokens_static(const dh_head_t *hd, const void *h, int M, int32_t *ids,
                                 float *top_logit, void *stream);

/* Synchronise `stream`, then read and clear the device error word of the
 * static scratch of draft_head_top_tokens_static on the current device
 * (DH_DEVERR_* bits; *err = 0 when nothing was recorded). As the first call
 * on a device, it looks up the array's address like that entry point. */
int draft_head_static_read_device_error(int *err, void *stream);

/* Self-test of the failure handling of the draft-step kernels (the pages have
 * no counterpart): a one-thread kernel waits for an event that nothing
 * produces and gives up after `rounds` tries, recording DH_DEVERR_TIMEOUT in
 * the error word of `ws` exactly as a draft step whose wait ran out does; the
 * context stays usable. kind 0: polls a word of the workspace header that
 * nothing writes (a bounded poll of global memory, the argmax hand-off's
 * wait); kind 1: waits on a shared-memory mbarrier that nothing arrives on
 * (the load pipeline's wait).
 * ws: a workspace of at least draft_head_quantize_workspace_bytes() bytes
 * (ws_bytes), or NULL for the static scratch of draft_head_top_tokens_static
 * on the current device (ws_bytes ignored); 1 <= rounds <= 2^22 (a draft
 * step's own limit). Read the result with draft_head_read_device_error
 * (draft_head_static_read_device_error for NULL). Errors: DH_ERR_ARG (kind,
 * rounds), DH_ERR_WORKSPACE. */
int draft_head_wait_probe(void *ws, size_t ws_bytes, int kind, unsigned int rounds, void *stream);

/* Synchronise `stream`, then read and clear the device error word of `ws`
 * (draft-step or quantiser workspace). *err = 0 when nothing was recorded. */
int draft_head_read_device_error(void *ws, int *err, void *stream);

/* Static description of a status code. */
const char *draft_head_status_string(int status);

/* DH_ABI_VERSION of the loaded library. */
int draft_head_abi_version(void);

/* The cudaError_t of the CUDA call or launch behind the calling thread's most
 * recent DH_ERR_CUDA (0 before any). If name is not NULL, *name points to the
 * error's static name (cudaGetErrorName). Host only; never touches the GPU. */
int draft_head_last_cuda_error(const char **name);

#ifdef __cplusplus
}
#endif

#endif /* DRAFTHEAD_H */
