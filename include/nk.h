/*
 * nk.h -- C ABI of libnk: paged KV cache append and paged attention on
 * NVIDIA GB300 (sm_103a).
 *
 * Source of the contract: the "Paged KV cache" maintainer design page of the
 * NInfer inference engine (typed growing KV pools, P = 64 token pages, block
 * tables, non-owning consumer views).  Section names below refer to that page
 * unless another page is named.
 *
 * Conventions for every call
 *  - Every pointer argument marked "device" points to GPU memory owned by the
 *    caller; libnk never allocates, frees or retains caller memory beyond the
 *    call (a pool handle borrows its plane pointers for its lifetime).
 *  - Calls that take a cudaStream_t (passed as void*) are asynchronous on that
 *    stream, never synchronize, and launch nothing when they return an error.
 *    NULL means the legacy default stream.
 *  - Return value: NK_OK (0) or a negative NK_ERR_* code; nk_last_error()
 *    then describes the failure (thread-local text).  No exception crosses
 *    the ABI.  Argument checks happen on the host before any launch, so an
 *    error return has no side effect.
 *  - Caller guarantees (consumer view section, "wrapper validates / caller
 *    guarantees"): every logical block a call may touch is mapped in its
 *    table row, reads stay below the frozen valid frontier, the table rows in
 *    use are not rewritten while the call is in flight.  The kernels still
 *    never access memory outside the pool when a guarantee is broken: a page
 *    id outside [0, M), a table row outside [0, C) or a position / frontier
 *    outside [0, L*P] is skipped (append) or read as page 0 / an empty row
 *    (attention), the affected results are undefined, and an NK_STATUS_* bit
 *    is recorded in the device status word (nk_status_read).
 *  - bf16 tensors are little-endian IEEE bfloat16; layouts are C order
 *    (row-major, last index fastest).
 */
#ifndef NK_H_
#define NK_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NK_PAGE_TOKENS 64 /* P: allocation granularity of every growing pool */

/* Return codes. */
enum {
  NK_OK = 0,
  NK_ERR_INVALID_ARG = -1, /* null pointer, bad enum, non-finite scale       */
  NK_ERR_SHAPE = -2,       /* B, T, Hq, head_dim or layer out of range        */
  NK_ERR_RANGE = -3,       /* page-group count M outside [M_min, M_max]       */
  NK_ERR_UNSUPPORTED = -4, /* profile / head_dim / GQA combination not built  */
  NK_ERR_ALIGN = -5,       /* pointer not 16-byte aligned                     */
  NK_ERR_CUDA = -6,        /* a CUDA runtime or driver call failed            */
  NK_ERR_WORKSPACE = -7    /* workspace smaller than required                 */
};

/* Bits of the device status word (nk_status_read). */
enum {
  NK_STATUS_PAGE_RANGE = 1,  /* a table entry was outside [0, M)             */
  NK_STATUS_FRONTIER = 2,    /* a position reached past L*P of its row       */
  NK_STATUS_TIMEOUT = 4      /* a bounded wait on a copy barrier ran out     */
};

/* KV profiles ("Paged KV cache" page, pool contents paragraph: BF16,
 * INT8-G64, FP8-E4M3FN-row256, NVFP4-G16 and the closed asymmetric K8V4 with
 * K = FP8-E4M3FN-row256 and V = NVFP4-G16).  Codec rules (the page leaves them
 * open; this library states them):
 *   BF16      codes = bf16 bits unchanged.
 *   INT8-G64  per 64 elements: s = min(fp16(fp32(amax/127)), 65504),
 *             q = clamp(RNE(x/s), -127, 127); s == 0 -> q = 0.
 *   FP8-row   per (token, head) row: s = min(fp16(fp32(amax/448)), 65504),
 *             c = E4M3FN RNE satfinite (x/s); s == 0 -> c = 0.
 *   NVFP4-G16 per 16 elements: s8 = E4M3FN RNE satfinite (fp32(amax/6)),
 *             c = E2M1 RNE satfinite (x/s8); s8 == 0 -> c = 0; element 2i in
 *             the low nibble of byte i.
 * Quotients are exact quotients rounded once; the sign bit of an E4M3/E2M1
 * code is the sign of its quotient.  A binary16 scale saturates at the
 * largest finite binary16 (65504) instead of becoming +inf, as the E4M3 /
 * E2M1 codes saturate: a group whose amax exceeds 127 * 65504 (INT8-G64) or
 * 448 * 65504 (FP8-row) keeps s = 65504 and its large elements clamp to the
 * extreme code, so every stored scale and every dequantized value is
 * finite. */
typedef enum {
  NK_BF16 = 0,
  NK_INT8_G64 = 1,
  NK_FP8_E4M3_ROW = 2,
  NK_NVFP4_G16 = 3,
  NK_K8V4 = 4
} nk_profile;

/* Plane order ("Paged KV cache" page, closed orders: page-major
 * [X, P, H, N_physical] for Main/MTP pools, head-major [X, P, N_physical, H]
 * for the draft pool).  Both are built: a (page group g, KV head h) tile of
 * 64 token rows starts at row (g * H + h) * 64 of a plane in page-major order
 * and at row (h * M + g) * 64 in head-major order. */
typedef enum { NK_PAGE_MAJOR = 0, NK_HEAD_MAJOR = 1 } nk_order;

/* Pool flags.  NK_POOL_CHECK_BOUNDS is accepted for callers that ask for
 * checked kernels; the range checks described above are always on. */
enum { NK_POOL_CHECK_BOUNDS = 1 };

/* Geometry of one typed growing pool (capacity section: S = max_context,
 * C = max_concurrency in 1..8, P = 64, L = ceil(S/P)). */
typedef struct {
  int32_t profile;         /* nk_profile                                     */
  int32_t num_layers;      /* >= 1                                           */
  int32_t num_kv_heads;    /* H >= 1                                         */
  int32_t head_dim;        /* D in {64, 128, 256}                            */
  int32_t max_context;     /* S >= 1                                         */
  int32_t max_concurrency; /* C in 1..8; block table has C rows of L entries */
  int32_t order;           /* nk_order                                       */
  int32_t flags;           /* NK_POOL_* bits                                 */
} nk_pool_desc;

typedef struct nk_pool nk_pool; /* opaque; borrows the caller's planes */

/* Version of this ABI (major * 10000 + minor * 100 + patch). */
int nk_version(void);

/* Text of the last error on this thread ("" when none).  Never NULL. */
const char* nk_last_error(void);

/* Plane inventory of one layer (physical layout section: code plane X = D,
 * INT8-G64 scale X = D/64, FP8-row scale X = 1, NVFP4 packed codes X = D/2
 * and scales X = D/16; PageBytes = sum of plane bytes per token * P).
 * Planes of a profile are ordered [K code, V code, K scale, V scale]; BF16
 * has only the first two.  Writes *n_planes (2 or 4) and, for each plane, its
 * byte size for M page groups (bytes[i] = X * elem_bytes * P * H * M) and its
 * bytes per token per head (row_bytes[i]; may be NULL).  Host only; no CUDA
 * call.  Errors: NK_ERR_INVALID_ARG, NK_ERR_UNSUPPORTED, NK_ERR_SHAPE. */
int nk_pool_plane_bytes(const nk_pool_desc* desc, int32_t M, int32_t* n_planes,
                        size_t bytes[4], size_t row_bytes[4]);

/* Capacity bounds (capacity section): *m_min = max(L, C), *m_max = C * L.
 * Host only. */
int nk_pool_capacity_bounds(const nk_pool_desc* desc, int32_t* m_min, int32_t* m_max);

/* Physical pages of the MTP backend pool ("Paged KV cache" page, physical
 * capacity of the selected speculative backend): the Main pool's M page
 * groups plus, for each of the C active rows, the pages of its provisional
 * lead over Main in one speculative round of draft window K:
 *   pages = M + C * ceil((K - 1) / 64).
 * The lead does not enlarge any row's logical capacity L.  Errors:
 * NK_ERR_INVALID_ARG (NULL), NK_ERR_RANGE (M, C or K < 1; result > INT32_MAX). */
int nk_pool_mtp_pages(int32_t M, int32_t C, int32_t draft_window, int32_t* pages);

/* Logical pages a row keeps mapped in one pool ("Paged KV cache" page, trim of
 * rejected speculative tails): ceil(max(committed, provisional) / 64).  The
 * mappings of later logical blocks may be released; the last partial page is
 * kept, and its bytes past the committed frontier are stale: no consumer reads
 * them (every kernel stops at its frontier) and the next append at the
 * frontier overwrites them.  Errors: NK_ERR_INVALID_ARG, NK_ERR_RANGE (< 0). */
int nk_pages_needed(int32_t committed_frontier, int32_t provisional_frontier, int32_t* pages);

/* Creates a pool handle over caller-owned planes.
 *   planes: host array of num_layers * n_planes device pointers, layer-major
 *           (planes[layer * n_planes + i]); each 16-byte aligned and at least
 *           nk_pool_plane_bytes(...).bytes[i] long.  Their contents are not
 *           touched; their addresses must stay valid and fixed for the
 *           handle's lifetime (graph-stable arguments section).
 *   M:      page groups, within [M_min, M_max] (capacity section).
 * Must be called with the device that owns the planes current; encodes the
 * TMA descriptors of every code plane.  The handle is freed by
 * nk_pool_destroy and owns no device memory.  Errors: NK_ERR_INVALID_ARG,
 * NK_ERR_UNSUPPORTED, NK_ERR_SHAPE, NK_ERR_RANGE, NK_ERR_ALIGN, NK_ERR_CUDA. */
int nk_pool_create(const nk_pool_desc* desc, int32_t M, void* const* planes, nk_pool** out);

int nk_pool_destroy(nk_pool* pool);

/* Growing-cache append with fused quantization (persistent codec named by the
 * page: "kv_cache_append"; translation paragraph of the consumer view
 * section).  For compact row b (0 <= b < B) and token t < count_b, where
 * count_b = counts ? counts[b] : T, the token goes to logical position
 * pos = write_pos[b] + t of table row table_rows[b]:
 *   g = block_tables[table_rows[b] * L + (pos >> 6)],  o = pos & 63,
 * and its K and V codes and scales of every KV head h are written at
 * base + d*nb0 + o*nb1 + h*nb2 + g*nb3 of the layer's planes.
 *   block_tables: device int32 [C][L];  table_rows, write_pos, counts: device
 *   int32 [B];  k, v: device bf16 [B][T][H][D] (16-byte aligned).
 * Writes only the addressed token rows.  Two appends that address the same
 * (g, o) in one call race.  Errors: NK_ERR_INVALID_ARG, NK_ERR_SHAPE
 * (B < 1 or B > C, T < 1, layer out of range), NK_ERR_ALIGN, NK_ERR_CUDA. */
int nk_paged_kv_append(nk_pool* pool, int32_t layer, const int32_t* block_tables,
                       const int32_t* table_rows, const int32_t* write_pos,
                       const int32_t* counts, const void* k, const void* v, int32_t B,
                       int32_t T, void* stream);

/* Workspace the decode call needs for (B, T, Hq) on the current device. */
int nk_decode_workspace_bytes(const nk_pool* pool, int32_t B, int32_t T, int32_t Hq,
                              size_t* bytes);

/* Compact-batch GQA decode / multi-query verify attention that reads the
 * pages in place through the block tables (consumer view section, batched
 * view with table_rows[B]; "no gather-to-contiguous copy").
 * Row b has valid length F_b = frontiers[b] (which already counts its T new
 * tokens); query token t of row b attends keys j <= F_b - T + t.  Query head
 * i uses KV head i / (Hq / H).  Scores s_j = softmax_scale * <q, K^_j>, with
 * K^ the dequantized keys;  out = softmax(s) V^ ;  lse = ln sum_j exp(s_j).
 *   q:    device bf16 [B][T][Hq][D];   out: device bf16 [B][T][Hq][D];
 *   lse:  device fp32 [B][T][Hq] or NULL;  a row with F_b - T + t < 0 gets
 *         out = 0, lse = -inf.
 *   workspace: device scratch of at least nk_decode_workspace_bytes bytes
 *         holding the split-K partials; no initialisation needed (two calls
 *         that share a workspace must not overlap).
 * Split-K over pages, then a log-sum-exp merge kernel launched right behind
 * (one CTA per row, KV head and 32 dims); no host synchronisation, so the
 * call can be captured in a CUDA graph (graph-stable arguments section).
 * Kernels are launched with programmatic stream serialization (they may start
 * while the previous kernel in the stream drains, and read nothing before it
 * completes).
 * R = T * Hq / H query rows per KV head: R <= 16 runs a warp-level tensor-core
 * kernel for every profile; 17 <= R <= 32 over FP8-row, NVFP4-G16 and K8V4
 * pools runs a 5th-generation tensor-core kernel (csrc/vdecode.cu), and over
 * BF16 and INT8-G64 pools the warp-level kernel at head_dim 64 and 128.
 * The split count per (row, KV head) is at most 32; at head_dim 64 and 128
 * the tensor-core kernel may take several splits per CTA.  Either way the
 * partials fit the workspace that nk_decode_workspace_bytes reports.
 * Keys enter the scores exactly (row and group scales multiply fp32 partial
 * scores).  In the warp-level kernel INT8-G64 and FP8-row values are f16
 * products code * scale * 2^K (relative error <= 2^-11 above f16's subnormal
 * range), K <= 0 lowered where needed so that no product overflows; in the
 * tensor-core kernel FP8-row value scales multiply the f16 softmax weights,
 * lifted by 2^K so that they stay finite and normal.  Either way 2^K is
 * removed before the output, so V of any magnitude is handled.
 * Errors: NK_ERR_INVALID_ARG, NK_ERR_SHAPE (Hq % H, B > C, T < 1),
 * NK_ERR_UNSUPPORTED (R > 32, or R > 16 at head_dim 256 over BF16 or
 * INT8-G64 pools), NK_ERR_ALIGN, NK_ERR_WORKSPACE, NK_ERR_CUDA. */
int nk_paged_decode_attention(const void* q, int32_t Hq, const nk_pool* pool, int32_t layer,
                              const int32_t* block_tables, const int32_t* table_rows,
                              const int32_t* frontiers, int32_t B, int32_t T,
                              float softmax_scale, void* out, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream);

/* nk_paged_kv_append followed by nk_paged_decode_attention in one launch: the
 * T new tokens of every row are written at positions F_b - T .. F_b - 1
 * (write_pos = frontiers - T), with the codec rules of nk_paged_kv_append,
 * and then attended together with the rest of the row.  The decode step of
 * the engine page's compact batch is exactly this pair ("Paged KV cache"
 * page: codes and scales are complete before the frontier is published;
 * "Engine architecture" page: compact decode batch).  Each CTA encodes the
 * new tokens whose pages it reads and orders those stores before its own TMA
 * reads of the pages, so no other kernel or host step is involved.
 *   k, v: device bf16 [B][T][H][D] (16-byte aligned); other arguments and
 *   the workspace contract as in nk_paged_decode_attention.
 * A row with F_b < T is rejected on the device (status NK_STATUS_FRONTIER,
 * nothing written, out = 0, lse = -inf).
 * Ordering: launched with programmatic stream serialization, the call reads
 * the block tables, table_rows, frontiers and the pool pages of earlier tokens
 * before it waits for the previous kernel in the stream (it overlaps that
 * kernel's tail); only q, k and v may be produced by that kernel.  After a
 * separate nk_paged_kv_append into the same rows, use nk_paged_decode_attention.
 * Errors: as nk_paged_decode_attention. */
int nk_paged_append_decode_attention(const void* q, int32_t Hq, nk_pool* pool, int32_t layer,
                                     const int32_t* block_tables, const int32_t* table_rows,
                                     const int32_t* frontiers, const void* k, const void* v,
                                     int32_t B, int32_t T, float softmax_scale, void* out,
                                     float* lse, void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ---- host replicas: logical-order packed pages and transfer runs ----------
 * "Paged KV cache" page, host replica section: a host replica holds the pages
 * of one address space in logical order, without device page ids or block
 * table holes; each packed page holds the whole grouped payload of the pool:
 * for layer l = 0..num_layers-1, for plane i (K code, V code, K scale, V
 * scale), the H * 64 * row_bytes[i] bytes of that page group in plane (l, i).
 * Transfers copy whole page payloads and merge runs of consecutive physical
 * ids (one strided copy per run, layer and plane). */

/* Bytes of one packed host page of `pool`. */
int nk_host_page_bytes(const nk_pool* pool, size_t* bytes);

/* Host helper: splits page_ids[0..n) (logical order) into runs of consecutive
 * physical ids; run r starts at logical page run_first[r] and has run_len[r]
 * pages.  run_first / run_len (each of n entries) may be NULL to count only.
 * Errors: NK_ERR_INVALID_ARG, NK_ERR_SHAPE (n < 0). */
int nk_page_runs(const int32_t* page_ids, int32_t n, int32_t* run_first, int32_t* run_len,
                 int32_t* n_runs);

/* Copies pages page_ids[0..n) (host int32, logical order) of every layer and
 * plane to `host` (n * nk_host_page_bytes bytes, packed as above; page-locked
 * memory makes the copies asynchronous on `stream`).  The caller keeps the
 * pages unchanged until the copies complete.  Errors: NK_ERR_INVALID_ARG,
 * NK_ERR_SHAPE, NK_ERR_RANGE (an id outside [0, M); nothing is copied),
 * NK_ERR_CUDA. */
int nk_pages_to_host(const nk_pool* pool, const int32_t* page_ids, int32_t n, void* host, void* stream);

/* The inverse: writes packed host pages into page groups page_ids[0..n) of
 * every layer and plane (a restore may target other physical pages than the
 * ones the replica came from).  Errors: as nk_pages_to_host. */
int nk_pages_from_host(nk_pool* pool, const int32_t* page_ids, int32_t n, const void* host, void* stream);

/* Size of the static device scratch of nk_paged_decode_attention_noalloc. */
#define NK_NOALLOC_SCRATCH_BYTES (32u << 20)

/* nk_paged_decode_attention for callers that cannot allocate device memory
 * (allocator callbacks, runtimes with a memory budget fixed at start-up,
 * loops that must never block on the driver's allocator).  The design page
 * has no counterpart: this is an interface choice of this library.
 * Same arguments, results and errors as nk_paged_decode_attention, without
 * the workspace: the split-K partials live in a static device array of
 * NK_NOALLOC_SCRATCH_BYTES (32 MiB) that every device that loads this entry
 * point keeps until the process exits.  The number of splits is lowered
 * until the partials fit; a call that does not fit even with one split per
 * (row, KV head) is rejected with NK_ERR_WORKSPACE before any launch.
 * The first call on a device (with that device current, which must be the
 * pool's device) looks up the array's device address; make it before any
 * stream capture.  That address is kept for the life of the process, so do
 * not use this entry point on a device after cudaDeviceReset (or any other
 * reset of its primary context): the module is loaded again there and the
 * kept address is stale.  All calls share the array, which keeps the last
 * call's contents (every slot a call reads it writes first).  Two calls that
 * overlap on the GPU race.  Calls no allocating routine. */
int nk_paged_decode_attention_noalloc(const void* q, int32_t Hq, const nk_pool* pool,
                                      int32_t layer, const int32_t* block_tables,
                                      const int32_t* table_rows, const int32_t* frontiers,
                                      int32_t B, int32_t T, float softmax_scale, void* out,
                                      float* lse, void* stream);

/* Workspace the prefill call needs (may be 0).  It depends on B, Tc, Hq, the
 * KV heads and D only, never on the pool's context length. */
int nk_prefill_workspace_bytes(const nk_pool* pool, int32_t B, int32_t Tc, int32_t Hq,
                               size_t* bytes);

/* Chunked prefill / replay attention through the block tables (every
 * profile; quantized pages are dequantized inside the tensor-core kernel,
 * page tile by page tile in shared memory, with no copy of the context
 * elsewhere.  The tiles hold FP8-row, NVFP4-G16 and K8V4 keys and values
 * and INT8-G64 keys exactly (an INT8-G64 key tile as two f16 tiles whose sum
 * is code times group scale); INT8-G64 values are rounded once to f16,
 * relative error <= 2^-11.  Softmax weights are f16 over quantized pools,
 * with FP8-row value scales applied under a power-of-two lift that keeps
 * them in f16's normal range for V of any magnitude, and bf16 over BF16
 * pools: relative error <= 2^-8 per weight, so there the output is within
 * 2^-8 of the attention over |V| of the exact one, beyond fp32 rounding).
 * Query i < chunk_len[b] of row b sits at logical position prefix_len[b] + i
 * and attends keys j <= prefix_len[b] + i; the chunk's own K/V must already
 * be appended.  Prefill work is proportional to prefix*S + S(S+1)/2 query-key
 * pairs ("Resource scheduling and context cache" page, machine cost model).
 *   q_chunk: device bf16 [B][Tc][Hq][D];  out: device bf16 [B][Tc][Hq][D]
 *   (rows i >= chunk_len[b] are not written);  lse: device fp32 [B][Tc][Hq]
 *   or NULL;  prefix_len, chunk_len: device int32 [B], chunk_len[b] <= Tc.
 *   workspace: nk_prefill_workspace_bytes bytes, zero-filled before its first
 *   use (every call leaves its counters at zero): when the launch splits each
 *   128-row tile over its pages to fill the last wave of SMs, the split
 *   partials and counters.
 * Errors as for decode; NK_ERR_UNSUPPORTED for D other than 64, 128 and 256,
 * or a GQA group that does not divide 128 or exceeds 16. */
int nk_paged_prefill_attention(const void* q_chunk, int32_t Hq, const nk_pool* pool,
                               int32_t layer, const int32_t* block_tables,
                               const int32_t* table_rows, const int32_t* prefix_len,
                               const int32_t* chunk_len, int32_t B, int32_t Tc,
                               float softmax_scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, void* stream);

/* Partial-tail copy-on-write of a Fork (Move/Fork section, worked example
 * F = 1000: 15 shared full pages, 40 tail columns copied to one private
 * page).  Copies token columns [0, ncols) of page group src into page group
 * dst in every plane of every layer; full pages are shared, never copied.
 * 0 <= ncols <= 64; src != dst; both in [0, M). */
int nk_page_copy_columns(const nk_pool* pool, int32_t src, int32_t dst, int32_t ncols,
                         void* stream);

/* Reads (and optionally clears) the device status word of the current device
 * (NK_STATUS_* bits set by kernels of pools created with
 * NK_POOL_CHECK_BOUNDS, and by bounded waits that ran out).  Synchronizes
 * `stream`. */
int nk_status_read(int32_t* status, int32_t clear, void* stream);

/* Self-test of the bounded waits (no counterpart on the design pages: the
 * pages leave failure handling of the consumer kernels open).  Every
 * pipeline wait of this library gives up after a wall-clock limit, records
 * NK_STATUS_TIMEOUT in the device status word and lets its kernel return, so
 * that a lost copy never hangs the GPU.  This call launches one kernel on
 * `stream` whose wait can never be satisfied (an mbarrier phase that expects
 * one more arrival than it gets; no copy is involved) and that gives up after
 * `limit_us` microseconds (1 .. 1000000).  Afterwards NK_STATUS_TIMEOUT is
 * set in the status word of the current device (nk_status_read), and, when
 * `waited_ns` is a device pointer, it receives the nanoseconds the wait took
 * (-1 if the wait had completed, which cannot happen).  Asynchronous; errors:
 * NK_ERR_INVALID_ARG for a limit outside the range, NK_ERR_CUDA on a launch
 * failure. */
int nk_selftest_bounded_wait(int32_t limit_us, long long* waited_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* NK_H_ */
