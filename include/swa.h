/*
 * swa.h -- C ABI of libswa: causal sliding-window attention with attention
 * sinks on NVIDIA B300 (sm_103a).
 *
 * The operation.  For a query at position i the keys it reads are the window
 * i-w+1 .. i (w cells including the current one) united with the g "sink"
 * positions 0 .. g-1, never a future key; every other key gets a score of
 * -inf before the softmax:
 *     O[i] = sum_j softmax_j(scale * q_i . k_j) v_j  over the allowed j.
 * Sources: "Sliding Window and Sparse Attention, from Longformer to CSA2",
 * sections 1 (attention, causal masking, prefill vs decode) and 2 (the window,
 * the rolling buffer, attention sinks); "Local and Sparse Attention: Reading
 * Fewer Token Positions", Figures 1 (window of w cells including the current
 * one, -inf masking), 2 (a key in the window and the designated set is read
 * once; no future key) and 4 (rolling cache).
 *
 * Conventions shared by every entry point.
 *  - Layouts are row-major and contiguous:
 *      prefill Q, O   [B][H][n][d]        K, V     [B][Hkv][n][d]
 *      decode  q, O   [B][H][d]           Kc, Vc   [B][Hkv][w+g][d]
 *      lse            [B][H][n] (prefill) or [B][H] (decode), fp32, natural log
 *    The rolling cache keeps position p in ring slot p mod w (slots 0..w-1)
 *    and, when p < g, also in sink slot w+p (slots w..w+g-1).
 *  - Grouped-query attention: query head h reads key/value head h / (H/Hkv);
 *    H must be a multiple of Hkv.
 *  - d is 64 or 128.  Element type bf16 (accumulation in fp32) or fp32.
 *  - All tensor pointers are device pointers owned by the caller, 16-byte
 *    aligned.  The library never frees caller memory.
 *  - Kernels launch on the calling thread's current CUDA device
 *    (cudaGetDevice); every pointer of a call and its stream must belong to
 *    that device.
 *  - Every launch is asynchronous on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  SWA_OK means "validated and enqueued".  A
 *    device-side wait that runs out of time marks the library's device status
 *    word and the kernel returns early; swa_get_device_status() reads and
 *    clears it.
 *  - Arguments are validated on the host before any launch; an invalid call
 *    enqueues nothing and returns SWA_ERR_INVALID_ARG or SWA_ERR_UNSUPPORTED.
 *  - Threads.  Every entry point may be called from several host threads at
 *    once.  The library's own state is small: the decode workspaces of
 *    swa_decode() (one per device and stream, see there), the fixed scratch
 *    array of swa_decode_noalloc() (one per device, shared by every call),
 *    the per-device status word and per-device launch settings.  Calls whose
 *    buffers are all the caller's (prefill, swa_decode_ex with a workspace of
 *    its own, append) never share memory with one another.  swa_decode() calls
 *    on different streams use different workspaces; calls on one stream are
 *    ordered by that stream.  swa_decode_noalloc() calls all share one array:
 *    calls whose kernels overlap on the GPU race and must be serialised by
 *    the caller (one stream, or events).
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A cudaStream_t, declared without pulling in the CUDA headers. */
typedef struct CUstream_st *swa_stream_t;

typedef enum {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = -1,    /* null/unaligned pointer, bad size or value   */
    SWA_ERR_UNSUPPORTED = -2,    /* valid but not built (e.g. d not 64 or 128)  */
    SWA_ERR_CUDA = -3,           /* a CUDA runtime/driver call failed           */
    SWA_ERR_DEVICE_TIMEOUT = -4, /* a kernel's bounded wait ran out (device)    */
    SWA_ERR_ALLOC = -5,          /* library workspace allocation failed         */
    SWA_ERR_WORKSPACE = -6,      /* caller workspace too small                  */
    SWA_ERR_DEVICE_BOUNDS = -7   /* a debug build's device bounds check failed  */
} swa_status;

typedef enum { SWA_BF16 = 0, SWA_F32 = 1 } swa_dtype;

/* Fixed attention patterns (swa_prefill_pattern). */
typedef enum {
    SWA_PATTERN_WINDOW = 0,   /* the last w positions plus the sinks 0..g-1       */
    SWA_PATTERN_DILATED = 1,  /* positions i, i-r, ..., i-(w-1)r                  */
    SWA_PATTERN_STRIDED = 2,  /* every position j <= i with (i - j) mod r == 0    */
    SWA_PATTERN_LANDMARK = 3  /* the window and sinks plus every j <= i, j mod r == 0 */
} swa_pattern;

/* ---------------------------------------------------------------------- */
/* Prefill: the whole prompt at once, block-sparse over BMxBN tiles.       */
/* ---------------------------------------------------------------------- */

/*
 * swa_prefill -- bf16 prefill ("Sliding Window and Sparse Attention, from
 * Longformer to CSA2", sections 1-2 and the block-sparsity note in section 4:
 * only the key tiles that meet the band or the sink columns are computed).
 *   Q [B][H][n][d], K, V [B][Hkv][n][d], O [B][H][n][d]: bf16, device.
 *   n >= 1, w >= 1, g >= 0, scale > 0 and finite (applied to q.k).
 * Runs the tcgen05/TMEM tensor-core kernel.  Returns SWA_OK or an error code.
 */
int swa_prefill(const void *Q, const void *K, const void *V, void *O,
                int B, int H, int Hkv, int n, int d, int w, int g, float scale,
                swa_stream_t stream);

/*
 * swa_prefill_ex -- as swa_prefill, with the element type chosen by `dtype`
 * (SWA_BF16: tensor-core kernel; SWA_F32: fp32 CUDA-core kernel, same
 * semantics) and an optional log-sum-exp output `lse` [B][H][n] fp32 (NULL to
 * skip): lse = log(sum_j exp(scale*q.k_j)) over the allowed keys (section 6 of
 * the same page: the log-sum-exp lets partial results be normalised jointly).
 */
int swa_prefill_ex(const void *Q, const void *K, const void *V, void *O, float *lse,
                   int B, int H, int Hkv, int n, int d, int w, int g, float scale,
                   swa_dtype dtype, swa_stream_t stream);

/*
 * swa_prefill_sink_logit -- swa_prefill_ex with a learned per-head attention
 * sink logit ("Sliding Window and Sparse Attention, from Longformer to CSA2",
 * section 6, stage 3: a per-head logit that absorbs probability mass when no
 * key is relevant).  For query head h the softmax gets one more entry, score
 * sink_logit[h] (natural-log units, the same as scale * q.k) with a zero value
 * vector:
 *     O[i] = sum_j e^{s_ij} v_j / (e^{sink_logit[h]} + sum_j e^{s_ij}),
 *     lse[i] = log(e^{sink_logit[h]} + sum_j e^{s_ij}).
 * sink_logit: device fp32 [H] (4-byte aligned) or NULL (then this is
 * swa_prefill_ex).  The token sinks of g are unaffected: both may be used.
 */
int swa_prefill_sink_logit(const void *Q, const void *K, const void *V, void *O, float *lse,
                           const float *sink_logit, int B, int H, int Hkv, int n, int d, int w,
                           int g, float scale, swa_dtype dtype, swa_stream_t stream);

/*
 * swa_prefill_pattern -- prefill under another fixed pattern, with the
 * layouts, outputs and sink logit of swa_prefill_sink_logit.  For query
 * position i the allowed keys j <= i are:
 *   SWA_PATTERN_WINDOW    i-w+1 <= j or j < g (swa_prefill_sink_logit itself;
 *                         r is ignored);
 *   SWA_PATTERN_DILATED   j = i - k r for k = 0 .. w-1 ("Sliding Window and
 *                         Sparse Attention, from Longformer to CSA2", section
 *                         2, dilated windows: the cost of a window of w, a
 *                         reach r times longer);
 *   SWA_PATTERN_STRIDED   (i - j) mod r == 0 (same page, section 4: the
 *                         Sparse Transformer's strided head; w is ignored);
 *   SWA_PATTERN_LANDMARK  i-w+1 <= j, or j < g, or j mod r == 0 ("Local and
 *                         Sparse Attention: Reading Fewer Token Positions",
 *                         Figure 2, right: positions designated at regular
 *                         intervals, each key read once).
 * r >= 1.  The dilated and strided patterns take no sinks: g must be 0
 * (SWA_ERR_UNSUPPORTED otherwise).  Both run as R = r independent prefills,
 * one per residue class i mod r, each over its own subsequence of rows; the
 * landmark pattern adds, per 128-row query tile, the key tiles of the
 * landmark positions that lie before its band.  Same dtypes and error
 * behaviour as swa_prefill_sink_logit.
 */
int swa_prefill_pattern(const void *Q, const void *K, const void *V, void *O, float *lse,
                        const float *sink_logit, int B, int H, int Hkv, int n, int d,
                        swa_pattern pattern, int w, int g, int r, float scale, swa_dtype dtype,
                        swa_stream_t stream);

/*
 * swa_prefill_chunk -- chunked prefill into the rolling cache: T new tokens
 * of each sequence at positions pos0[b] .. pos0[b]+T-1 attend, with the
 * window and sink rule above, to the keys the rolling cache holds for the
 * positions before pos0[b] and to their own keys ("Sliding Window and Sparse
 * Attention, from Longformer to CSA2", section 1: prefill reads many
 * positions at once; section 2: the rolling buffer and the sinks).  This is
 * the step that takes a long prompt into the cache piece by piece.
 *   Q, O [B][H][T][d]; k_new, v_new [B][Hkv][T][d] (the chunk's keys and
 *   values); Kcache, Vcache [B][Hkv][w+g][d] holding every position before
 *   pos0[b] that the rolling cache keeps (appended with swa_cache_append);
 *   pos0: device int32 [B], >= 0; lse [B][H][T] fp32 or NULL; sink_logit
 *   [H] fp32 or NULL (as in swa_prefill_sink_logit).  dtype: SWA_BF16
 *   (tensor cores) or SWA_F32.
 * append = 0: the cache is only read (append the chunk afterwards with
 * swa_cache_append).  append != 0: after the keys are laid out in the
 * workspace, the chunk is written into Kcache/Vcache exactly as
 * swa_cache_append would write it, in stream order, so one call leaves the
 * cache holding positions up to pos0[b]+T-1 for the next chunk or decode step;
 * the attention itself reads the workspace copy and so sees the cache as it
 * was before the call.  workspace: caller-
 * owned device memory of at least swa_prefill_chunk_workspace_bytes(...)
 * bytes (16-byte aligned, no initialisation needed), where the kernel lays
 * out each sequence's keys in position order before the tensor-core pass.
 */
size_t swa_prefill_chunk_workspace_bytes(int B, int Hkv, int T, int d, int w, int g,
                                         swa_dtype dtype);
int swa_prefill_chunk(const void *Q, const void *k_new, const void *v_new, void *Kcache,
                      void *Vcache, const int32_t *pos0, void *O, float *lse,
                      const float *sink_logit, int B, int H, int Hkv, int T, int d, int w, int g,
                      float scale, int append, swa_dtype dtype, void *workspace,
                      size_t workspace_bytes, swa_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Decode: one query token per sequence against the rolling cache.         */
/* ---------------------------------------------------------------------- */

/*
 * swa_decode -- bf16 single-token decode ("Sliding Window and Sparse
 * Attention, from Longformer to CSA2", section 1: decode streams the cache
 * from HBM; section 2: the rolling buffer and sinks).  The query of sequence
 * b is at position pos[b] (device int32 [B], pos >= 0) and its own key/value
 * must already be in the cache (swa_cache_append).  Slots whose position is
 * not yet written (pos < w-1) and sink slots of positions still inside the
 * window are not read.
 *   q [B][H][d], Kcache, Vcache [B][Hkv][w+g][d], O [B][H][d]: bf16, device.
 *   Any group size G = H/Hkv: the kernels score up to 8 heads of a group per
 *   pass over the cache rows; a larger group is split into ceil(G/8) equal
 *   sub-groups that stream the same rows side by side.
 * Split-K over the cached keys, then a log-sum-exp merge: a first kernel cuts
 * the cache rows of all (sequence, kv head) pairs, laid end to end, into equal
 * contiguous shares, one per CTA of a single resident wave, and writes one
 * partial (max, sum, unnormalised output) per share and pair; a second kernel
 * merges them.  Uses a library-owned workspace, one per (device, stream)
 * (per calling thread too for cudaStreamPerThread), so calls on different
 * streams may overlap safely.  A workspace grows on demand (cudaMalloc when a
 * stream first needs more, so make the first call of a size on a stream
 * outside stream capture); an outgrown buffer is kept, not freed, until the
 * process exits, because kernels or captured graphs may still use it.  A
 * stream's workspace also outlives the stream (the library is not told when a
 * stream is destroyed): a program that creates many short-lived streams should
 * call swa_decode_ex with a workspace of its own.  Returns SWA_ERR_ALLOC,
 * enqueuing nothing, if that allocation fails.
 */
int swa_decode(const void *q, const void *Kcache, const void *Vcache, const int32_t *pos,
               int B, int H, int Hkv, int d, int w, int g, float scale, void *O,
               swa_stream_t stream);

/* Bytes of workspace swa_decode_ex needs for these sizes and `num_splits`
 * (0 = the split count the library would choose). */
size_t swa_decode_workspace_bytes(int B, int H, int Hkv, int d, int w, int g, int num_splits);

/*
 * swa_decode_ex -- as swa_decode with the element type `dtype`, an optional
 * lse [B][H] fp32 output (NULL to skip), a split count `num_splits` (0 =
 * automatic, one resident wave of CTAs; n in 1..1024 = n*B*Hkv CTAs, about n
 * shares per (sequence, kv head)) and a caller-owned device workspace of
 * `workspace_bytes` >= swa_decode_workspace_bytes(...) (16-byte aligned; its
 * contents need no initialisation).  Nothing is allocated.
 */
int swa_decode_ex(const void *q, const void *Kcache, const void *Vcache, const int32_t *pos,
                  int B, int H, int Hkv, int d, int w, int g, float scale, void *O,
                  float *lse, swa_dtype dtype, int num_splits, void *workspace,
                  size_t workspace_bytes, swa_stream_t stream);

/*
 * swa_decode_sink_logit -- swa_decode_ex with the learned per-head sink
 * logit of swa_prefill_sink_logit (device fp32 [H] or NULL), applied in the
 * log-sum-exp merge of the split results.
 */
int swa_decode_sink_logit(const void *q, const void *Kcache, const void *Vcache,
                          const int32_t *pos, const float *sink_logit, int B, int H, int Hkv,
                          int d, int w, int g, float scale, void *O, float *lse, swa_dtype dtype,
                          int num_splits, void *workspace, size_t workspace_bytes,
                          swa_stream_t stream);

/*
 * swa_cache_append -- rolling-buffer scatter ("Sliding Window and Sparse
 * Attention, from Longformer to CSA2", section 2: position i overwrites slot
 * i mod w; "Local and Sparse Attention: Reading Fewer Token Positions",
 * Figure 4).  Writes T new tokens k_new, v_new [B][Hkv][T][d] of sequence b at
 * positions pos0[b] .. pos0[b]+T-1 (pos0: device int32 [B], 0 <= pos0[b] <=
 * INT32_MAX - T; a sequence whose pos0[b] is outside that range is left
 * untouched and marks the device status word, which swa_get_device_status()
 * then reports as SWA_ERR_INVALID_ARG): position p
 * goes to ring slot p mod w and, if p < g, also to sink slot w+p.  When T > w
 * only the last w positions are written to the ring (earlier ones would be
 * overwritten anyway); sink slots are written for every p < g.
 * Kcache, Vcache [B][Hkv][w+g][d] of `dtype`, device.
 */
int swa_cache_append(void *Kcache, void *Vcache, const void *k_new, const void *v_new,
                     const int32_t *pos0, int T, int B, int Hkv, int d, int w, int g,
                     swa_dtype dtype, swa_stream_t stream);

/*
 * swa_decode_noalloc -- swa_decode for callers that cannot allocate device
 * memory: plugins and embedded runtimes handed only their input and output
 * buffers, processes whose device memory belongs to another allocator, and
 * latency-critical loops where cudaMalloc/cudaFree (and the synchronisation
 * a free implies) are not allowed.  The pages have no counterpart: this is an
 * interface variant, not part of the method.
 * Same arguments, semantics and result as swa_decode (bf16).  It allocates
 * nothing: the split-K partial results go to a fixed array of
 * SWA_NOALLOC_SCRATCH_BYTES in the library's own device memory, present on
 * every GPU that loads the library until the process exits.  Sizes whose
 * workspace (swa_decode_workspace_bytes(..., 0)) exceeds that array return
 * SWA_ERR_WORKSPACE and enqueue nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress) with that device current;
 * make that first call before any stream capture.  All calls share the array
 * and it keeps the last call's contents (nothing needs to start at zero);
 * calls whose kernels overlap on the GPU race and must be serialised.
 */
#define SWA_NOALLOC_SCRATCH_BYTES (4u << 20)
int swa_decode_noalloc(const void *q, const void *Kcache, const void *Vcache, const int32_t *pos,
                       int B, int H, int Hkv, int d, int w, int g, float scale, void *O,
                       swa_stream_t stream);

/* ---------------------------------------------------------------------- */
/* Host helpers (no GPU needed).                                           */
/* ---------------------------------------------------------------------- */

/* Number of (query, key) connections of one head over n positions
 * ("Local and Sparse Attention: Reading Fewer Token Positions", Figure 1: 21
 * for n=8, w=3; 36 for full causal).  Returns -1 on invalid input. */
int64_t swa_count_pairs(int64_t n, int64_t w, int64_t g);

/*
 * Tile classes the prefill kernels use: for query tile qt (rows qt*BM ..) and
 * key tile kt (columns kt*BN ..), cls[qt*n_kt + kt] = 0 skipped, 1 partial
 * (element mask applied), 2 full, with n_qt = ceil(n/BM), n_kt = ceil(n/BN);
 * `cap` is the number of int32 elements at `cls` (host memory).  Only rows < n
 * exist; columns >= n are blocked.  Returns SWA_OK or SWA_ERR_INVALID_ARG.
 */
int swa_enumerate_tiles(int64_t n, int64_t w, int64_t g, int BM, int BN, int32_t *cls,
                        size_t cap);

/*
 * Landmark tiles of the landmark pattern (swa_prefill_pattern with
 * SWA_PATTERN_LANDMARK; "Local and Sparse Attention: Reading Fewer Token
 * Positions", Figure 2, right).  The landmarks 0, r, 2r, ... form a list
 * indexed by m (position r*m); for query tile qt (rows qt*BM ..) and landmark
 * tile lt (landmarks lt*BN ..), cls[qt*n_lt + lt] = 0 not visited, 1 partial,
 * 2 full, n_lt = ceil(ceil(n/r)/BN).  These tiles carry only the landmarks a
 * row reads outside its band and sinks (g <= r*m <= i-w); the band and sink
 * tiles are those of swa_enumerate_tiles.  Landmarks past the list count as
 * blocked.  Host memory, `cap` int32 elements.  Returns SWA_OK or
 * SWA_ERR_INVALID_ARG.
 */
int swa_enumerate_landmark_tiles(int64_t n, int64_t w, int64_t g, int64_t r, int BM, int BN,
                                 int32_t *cls, size_t cap);

/*
 * The key list a chunked prefill (swa_prefill_chunk) builds for a chunk of T
 * tokens at positions pos0 .. pos0+T-1: position[r] is the token position
 * whose key sits at index r of the list, or -1 for a padding row (the rows
 * between the sinks and the window that align the chunk's queries with the
 * 128-row tiles, and the rows past the list's end); query t of the chunk sits
 * at index t + *query_offset.  The prefill kernels read index j for query
 * index i when j <= i and (j >= i-w+1 or j < g).  `position` is host memory of
 * `cap` int64 elements.  Returns the number of rows written (the workspace
 * rows of swa_prefill_chunk_workspace_bytes), or SWA_ERR_INVALID_ARG (also
 * when the list would exceed `cap` or INT32_MAX rows; nothing is written then).
 */
int swa_chunk_key_positions(int64_t pos0, int w, int g, int T, int64_t *position, size_t cap,
                            int32_t *query_offset);

/* Where the rolling cache keeps position p: *ring_slot = p mod w,
 * *sink_slot = w+p if p < g else -1.  Returns SWA_OK, or SWA_ERR_INVALID_ARG
 * if p < 0, w < 1, g < 0, w + g > INT32_MAX or an output pointer is null. */
int swa_cache_slot(int64_t p, int w, int g, int32_t *ring_slot, int32_t *sink_slot);

/* ---------------------------------------------------------------------- */
/* Status and diagnostics.                                                  */
/* ---------------------------------------------------------------------- */

/* Synchronises `stream`, then reads and clears the current device's status
 * word: SWA_OK; SWA_ERR_DEVICE_TIMEOUT if a kernel's bounded wait ran out;
 * SWA_ERR_INVALID_ARG if a decode, append or chunked prefill met a position
 * outside its range (negative, or past INT32_MAX); SWA_ERR_CUDA if a CUDA call
 * failed. */
int swa_get_device_status(swa_stream_t stream);

/*
 * swa_debug_prefill_walk -- a diagnostic with no counterpart on the pages: runs
 * swa_prefill_pattern (bf16, tensor-core kernels; no lse, no sink logit) and
 * logs every key tile the kernels' producers load, so that a test can compare
 * the tile walk the kernels actually take with the tile set the method
 * defines ("Sliding Window and Sparse Attention, from Longformer to CSA2",
 * section 4: only the key tiles that meet the band or the sinks are read).
 * log: device int32, 16-byte aligned, 8 + 8 * log_entries elements; log[0]
 * counts the tiles loaded (entries past log_entries are counted, not stored);
 * entry e at log[8 + 8e] is {work item rank, sequence b, kv head, unit, q tile,
 * residue class, first key index of the tile, flags}.  The unit is the head
 * pair (even groups: heads kvh*G + 2u, +1), the q-tile pair of head kvh*G + u
 * (odd groups, window and sinks: q tiles 2*qtile and 2*qtile + 1), or the head
 * kvh*G + u (odd groups under the other patterns); q tiles and key indices
 * count 128-row tiles and rows of the residue class's subsequence for the
 * dilated and strided patterns, and landmark-list entries for landmark tiles.
 * flags: 1 the tile needs no element mask, 2 a landmark tile.  Returns as
 * swa_prefill_pattern.
 */
int swa_debug_prefill_walk(const void *Q, const void *K, const void *V, void *O, int B, int H,
                           int Hkv, int n, int d, swa_pattern pattern, int w, int g, int r,
                           float scale, int32_t *log, int64_t log_entries, swa_stream_t stream);

/*
 * swa_debug_prefill_cta_pairs -- an alternative kernel for swa_prefill_ex
 * (bf16, window path) with no counterpart on the pages: the tile loop of the
 * default kernel on clusters of two CTAs that share each tensor-core MMA
 * (tcgen05 cta_group::2, M = 256), so that each SM reads half of the K and V
 * operands.  It computes the same output (and LSE, if lse is not null) as
 * swa_prefill_ex; it measured slower than the default kernel on this build's
 * workloads and is kept as a tested alternative, not used by the other entry
 * points.  Arguments, layouts and errors as swa_prefill_ex (dtype bf16), plus
 * SWA_ERR_UNSUPPORTED unless d == 128, H / Hkv is even and H % 4 == 0.
 */
int swa_debug_prefill_cta_pairs(const void *Q, const void *K, const void *V, void *O, float *lse,
                                int B, int H, int Hkv, int n, int d, int w, int g, float scale,
                                swa_stream_t stream);

/*
 * swa_debug_inject_stall -- a test aid with no counterpart on the pages; it
 * lets a test run the kernels' timeout path without faulting or hanging the
 * GPU.  The next launch of the chosen kind on the current device leaves out
 * its first key/value copy and gives each of its bounded waits `wait_ns`
 * nanoseconds instead of 2 s:
 *   kind 1 (SWA_STALL_PREFILL): the next bf16 prefill launch (swa_prefill*,
 *           swa_prefill_pattern, the attention of swa_prefill_chunk);
 *   kind 2 (SWA_STALL_DECODE):  the next decode split pass (swa_decode*).
 * A wait of that launch then runs out: the kernel stops early, waits for the
 * copies it did start, frees its tensor memory, and marks the device status
 * word, so swa_get_device_status() returns SWA_ERR_DEVICE_TIMEOUT.  That
 * launch's outputs are unspecified; later launches are unaffected.  The
 * setting is used once; kind 0 cancels a pending one.  wait_ns must be in
 * [1e5, 2e9].  Returns SWA_OK, SWA_ERR_INVALID_ARG or SWA_ERR_CUDA.
 */
#define SWA_STALL_PREFILL 1
#define SWA_STALL_DECODE 2
int swa_debug_inject_stall(int kind, int64_t wait_ns);

/*
 * Debug builds.  The library can be built with SWA_DEBUG defined
 * (libswa_debug.so beside libswa.so).  Its kernels then check, before each
 * global store they make and each index they derive from the tile walk, that
 * the index lies inside its buffer or range (output rows, LSE entries, decode
 * partials, cache slots, chunk key-list rows, key tiles, work items).  A check
 * that fails sets a bit in the device status word, so swa_get_device_status()
 * returns SWA_ERR_DEVICE_BOUNDS, and the store it guards is skipped; nothing
 * traps.  Product builds compile no checks and never return that status.
 *
 * swa_debug_shrink_bounds -- a test aid for debug builds, with no counterpart
 * on the pages: the next bf16 prefill launch on the current device checks its
 * output rows against a limit one row short of the real one, so the last
 * output row of the last head of the last sequence fails its check and is not
 * written.  Returns SWA_OK in a debug build, SWA_ERR_UNSUPPORTED in a product
 * build (which has no checks), SWA_ERR_CUDA if no device is current.
 */
int swa_debug_shrink_bounds(void);

/* A static string naming a swa_status value. */
const char *swa_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int swa_version(void);

/*
 * swa_selftest_umma -- diagnostic with no counterpart on the pages: checks the
 * tensor-core operand encodings the prefill kernel relies on, on one tile.
 *   A [128][128] bf16 (row-major), Bk [128][128] bf16 (row-major, read as
 *   N x K), Bn [128][128] bf16 (row-major, read as K x N), device.
 *   D1 = A . Bk^T with both operands from shared memory;
 *   D2 = A . Bn with A staged through tensor memory and Bn N-contiguous.
 *   D1, D2 [128][128] fp32, device.  One CTA.  Returns SWA_OK if enqueued.
 */
int swa_selftest_umma(const void *A, const void *Bk, const void *Bn, float *D1, float *D2,
                      swa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
