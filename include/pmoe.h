/*
 * pmoe.h -- C ABI of the paged fused-MoE layer forward for GB300 (sm_103a).
 *
 * The operation (Rimuru, paper-daily.com/en, section "Expert weights are scattered across
 * pages. How does the kernel read them?"): a fused MoE layer whose expert weights are not
 * stored contiguously.  Cached experts sit in pages of one shared page pool, experts copied in
 * for this step sit in a slot of one of two alternating load buffers, and the kernel takes, per
 * expert, where it is -- a page number or a buffer slot.  Gate (W1) and up (W3) projections of
 * an expert occupy one page each and the kernel picks the page by whether the output column n
 * is in the first or the second half; the element address is
 *
 *     addr_e(n, t) = B_P + p_e(n) * f * d + (n mod f) * d + t
 *
 * so the page lookup happens once per output tile and reads inside a page use fixed strides.
 * No contiguous copy of any expert is made.  Section "The adjuster": an expert takes three
 * pages, W1 (gate), W3 (up) and W2 (down projection).
 *
 * Conventions shared by every call below
 *   bf16       IEEE bfloat16 bit patterns (uint16 storage).
 *   page       f*d bf16 elements.  W1/W3 pages are [f rows][d cols] row-major (row n = output
 *              column n of the gate / up projection).  A W2 page is [d rows][f cols] row-major.
 *   pool       `num_pages` consecutive pages starting at `page_pool` (device memory).
 *   load buf   load_buf[b] holds `slots_per_buffer` slots; slot s holds the expert's W1, W3, W2
 *              pages back to back, matrix j at element offset (3*s + j) * f * d.
 *   page_table int32 [E + S][3] (device): pages of W1, W3, W2 for each routed expert e < E and
 *              each shared-expert chunk E + s (s < S; always pool-resident).
 *   buf_slot   int32 [E] (device): -1 = pool-resident (use page_table[e]); otherwise
 *              b * slots_per_buffer + s = slot s of load buffer b (b in {0, 1}); -2 = absent
 *              (see pmoe_copy_in_missing; an error if a token routes to it).
 *   shared     the shared expert of intermediate size S*f is split into S chunks of width f;
 *              chunk s is the expert E + s with weight 1 on every token.
 *   ownership  the caller owns every buffer: pool, load buffers, tables, activations, outputs,
 *              workspace, pinned host memory, streams and events.  The library allocates only
 *              in pmoe_plan_create (the plan object and one block of device words: the error
 *              word and the fused decode kernel's barrier words, tile counters and ready words,
 *              2 KB + 12 bytes per f/64 columns of every expert) and frees it in
 *              pmoe_plan_destroy.  Forward calls allocate nothing and never synchronise the host.
 *   errors     argument checks are synchronous and return a status.  Table contents are checked
 *              on the device: an out-of-range page or slot of an expert that the routing
 *              activates sets the plan's device error word (read it with pmoe_get_device_error)
 *              and the tiles of that expert are skipped; the output is then undefined.  No call
 *              traps, asserts or spins on the device.
 *   streams    every device step of a call is enqueued on the stream given; cudaStream_t and
 *              cudaEvent_t values are passed as pmoe_stream_t / pmoe_event_t.
 */
#ifndef PMOE_H
#define PMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pmoe_stream_t; /* = cudaStream_t */
typedef struct CUevent_st* pmoe_event_t;   /* = cudaEvent_t */

typedef enum {
    PMOE_OK = 0,
    PMOE_ERR_INVALID_ARG = 1, /* a size, pointer or flag is out of range */
    PMOE_ERR_PAGE_OOB = 2,    /* device error word: a page index outside [0, num_pages) */
    PMOE_ERR_SLOT_OOB = 3,    /* device error word: a buffer slot outside [0, 2*slots) */
    PMOE_ERR_UNSUPPORTED = 4, /* shape the kernels do not cover (see pmoe_plan_create) */
    PMOE_ERR_CUDA = 5,        /* a CUDA runtime call failed; pmoe_last_error() has the text */
    PMOE_ERR_TIMEOUT = 6,     /* pmoe_wait_event gave up */
    PMOE_ERR_WORKSPACE = 7    /* workspace too small for this call */
} pmoe_status;

/* One MoE layer's shape. */
typedef struct {
    int32_t d;                 /* hidden size; multiple of 64 */
    int32_t f;                 /* per-expert intermediate size; multiple of 128 */
    int32_t num_experts;       /* E routed experts, 1..1024 */
    int32_t top_k;             /* k, 1..min(E, 16) */
    int32_t renormalize;       /* 1: divide the k routing weights by their sum */
    int32_t num_shared_chunks; /* S >= 0; shared intermediate size S*f; E + S <= 1024, k + S <= 64 */
    int32_t slots_per_buffer;  /* expert_offload_limit: slots in each of the two load buffers */
} pmoe_layer_desc;

typedef struct pmoe_plan* pmoe_plan_t;

/* Kernel families a forward call may use (pmoe_plan_set_path). */
typedef enum {
    PMOE_PATH_AUTO = 0,   /* SLICE up to 16 tokens while no routing leaves an SM more than
                             10 MiB of weights; else FUSED up to 32 tokens (E <= 128) or 16 tokens
                             (E > 128); above, by routed tokens per expert T*k/E: <= 24
                             (and T <= 320) TC_DECODE, >= 64 TC2 when E <= 128, else TC */
    PMOE_PATH_STREAM = 1, /* weight-streaming kernels (decode sizes; CUDA cores) */
    PMOE_PATH_TC = 2,     /* tcgen05 tensor-core grouped GEMMs, 128 tokens per tile (large T) */
    PMOE_PATH_TC_DECODE = 3, /* tcgen05 with weight rows on the MMA's M side and 16..128 tokens
                                on N: weight streaming for small token counts */
    PMOE_PATH_TC2 = 4,      /* 128-token blocks, taken two at a time per expert by CTA pairs
                               (tcgen05 cta_group::2, 256x256 tiles); an expert's odd last
                               block runs in the same pair kernel with the weights on the MMA's
                               M side and its 128 tokens on N */
    PMOE_PATH_FUSED = 5,    /* T <= 32 only: the whole layer in one persistent tcgen05 kernel
                               (one CTA per SM) whose weight streams are split evenly over the
                               SMs; see moe_paged_forward for what it requires of the caller */
    PMOE_PATH_SLICE = 6     /* T <= 16 only: the whole layer in one persistent tcgen05 kernel
                               whose CTAs each own whole 64-column tiles of the intermediate
                               dimension (gate/up, SiLU-and-mul and their slice of the down
                               projection, no cross-CTA hand-off before the final sum); refused
                               (PMOE_ERR_UNSUPPORTED) when a routing could leave more than 12
                               tiles per SM; same caller requirements as PMOE_PATH_FUSED */
} pmoe_path;

/* Text of a status; never NULL. */
const char* pmoe_status_string(pmoe_status s);
/* Last error message of the calling thread (empty string if none). */
const char* pmoe_last_error(void);

/* Create a plan for one layer over a page pool and two load buffers (device pointers, each
 * 16-byte aligned; load buffers may be NULL when slots_per_buffer == 0).  Builds the TMA tensor
 * maps that view the pool as rows [num_pages*f, d] (W1/W3 pages) and [num_pages*d, f] (W2
 * pages), and each load buffer likewise, on the current device; allocates the device error
 * word.  The pool and the buffers must outlive the plan.  *out receives the plan. */
pmoe_status pmoe_plan_create(const pmoe_layer_desc* desc, const void* page_pool, int64_t num_pages,
                             const void* load_buf0, const void* load_buf1, pmoe_plan_t* out);
pmoe_status pmoe_plan_destroy(pmoe_plan_t plan);
/* Force a kernel family (tests, benchmarks); PMOE_PATH_AUTO restores the default. */
pmoe_status pmoe_plan_set_path(pmoe_plan_t plan, int32_t path);

/* The kernel family (pmoe_path) the plan's last forward call ran, how many steps the measurement
 * hook brackets (n_steps: events 0..n_steps are recorded) and how many kernels it launched
 * (zeros before the first call). */
pmoe_status pmoe_plan_last_run(pmoe_plan_t plan, int32_t* path, int32_t* n_steps,
                               int32_t* n_launches);

/* Measurement hook: while set, each forward call records events[i] on its stream right before
 * launching its i-th kernel and events[n_kernels] after the last one (at most n events are
 * recorded), so elapsed times between consecutive events are per-kernel durations.  The kernel
 * order is: routing, sort-and-pad, [row gather,] gate/up GEMM, down GEMM, combine, where for
 * T <= 128 routing and sort-and-pad are one kernel; the fused and column-slice decode paths are one
 * kernel each.  NULL entries
 * are skipped (to bracket one kernel only).  The caller owns the events; n = 0 (or events = NULL)
 * turns the hook off.  At most 16 events. */
pmoe_status pmoe_plan_set_profile_events(pmoe_plan_t plan, const pmoe_event_t* events, int32_t n);

/* Bytes of device workspace a forward call with up to max_tokens tokens needs (256-aligned
 * start required).  0 on invalid arguments. */
size_t pmoe_workspace_size(const pmoe_layer_desc* desc, int32_t max_tokens);

/* The layer forward.
 *   hidden        bf16 [T][d] (device)
 *   router_logits fp32 [T][E] (device); finite values
 *   top_k         must equal desc->top_k (the pages' signature carries it per call)
 *   page_table    int32 [E+S][3], buf_slot int32 [E] (device; see the conventions above)
 *   out           bf16 [T][d] (device); must not alias any input
 *   workspace     >= pmoe_workspace_size(desc, T) bytes of device memory, 256-byte aligned
 * Steps, all on `stream`: top-k softmax routing; stable sort of (token, slot) pairs by expert
 * with padding to the GEMM block size; page resolution and validation; gate/up GEMM with the
 * SiLU-and-mul epilogue; down GEMM; weighted top-k combine plus the shared expert.
 * out[t] = bf16( sum_j w[t,j] * y_{t,ids[t,j]} + sum_s y_{t,E+s} ), summed in that order.
 * The call neither allocates nor synchronises, so it can be captured in a CUDA graph; the
 * captured launches keep the addresses of this call's buffers and workspace.
 * Kernels are launched with programmatic dependent launch: a kernel may start while the
 * previous kernel of the stream is finishing, and before it waits for that kernel it already
 * reads the page pool, the load buffers, page_table and buf_slot (never hidden, logits or the
 * workspace).  So those four must not be written by a kernel of the same stream that triggers
 * its dependents early (no kernel of this library writes them; ordinary kernels and copies are
 * complete before the next launch starts).
 * The fused and column-slice decode paths (T <= 32, T <= 16) synchronise their CTAs through words
 * that the plan owns, so forward calls of one plan must not overlap on the GPU (the plan's error
 * word is shared the same way).  Their waits give up after about 2 s with PMOE_ERR_TIMEOUT in the error word (only if the
 * GPU cannot hold one CTA per SM for this call, e.g. when other work occupies SMs indefinitely);
 * reading the error word with clear != 0 resets the plan's words for the next call. */
pmoe_status moe_paged_forward(pmoe_plan_t plan, const void* hidden, int32_t T,
                              const float* router_logits, int32_t top_k, const int32_t* page_table,
                              const int32_t* buf_slot, void* out, void* workspace,
                              size_t workspace_bytes, pmoe_stream_t stream);

/* Where the plan's last forward call (moe_paged_forward or moe_contig_forward, with T tokens)
 * left its routing and sort state in its workspace, so that a test can read back what the kernels
 * of that very call computed and compare it with an independent implementation.  Each field is a
 * byte offset into that call's workspace, or -1 when the call's kernel family does not write the
 * array.  The contents stay valid until the workspace is reused.  PMOE_ERR_INVALID_ARG when T is
 * not the token count of the plan's last forward call.  Host only: no device access. */
typedef struct {
    int32_t path;          /* pmoe_path the call ran */
    int32_t tokens;        /* its T */
    int32_t block_m;       /* rows per sorted block; 0 on the fused and column-slice paths, which
                              sort nothing */
    int32_t top_k;         /* k */
    int64_t ids;           /* int32 [T][k]: the k experts of each token, largest logit first
                              (fused and column-slice paths: CTA 0's routing, every CTA routes
                              the same way) */
    int64_t weights;       /* fp32 [T][k]: their routing weights */
    int64_t sorted_ids;    /* int32 [n_padded]: the pair in each sorted row (pads hold T*(k+S)) */
    int64_t block_expert;  /* int32 [n_padded / block_m]: the expert of each block */
    int64_t inv;           /* int32 [T*(k+S)]: the sorted row of each pair */
    int64_t meta;          /* int32 [16]: [0] n_padded (sorting paths), [1] work units and [2] of
                              them single blocks (CTA-pair path), [3] active slots (fused and
                              column-slice paths) */
    int64_t block_rows;    /* int32 [n_padded / block_m]: valid rows of each block (PMOE_PATH_TC,
                              PMOE_PATH_TC_DECODE) */
    int64_t units;         /* int32 [meta[1]][4]: CTA-pair work units {first block << 1 | single
                              block, expert, W1 location, W3 location}, location = map << 29 | page
                              with map 0 pool, 1 + b load buffer b (PMOE_PATH_TC2) */
    int64_t active;        /* int32 [meta[3]]: the expert of each active slot, shared chunks
                              E..E+S-1 first, then the routed experts in ascending id (fused and
                              column-slice paths) */
} pmoe_routing_view;
pmoe_status pmoe_plan_routing_view(pmoe_plan_t plan, int32_t T, pmoe_routing_view* out);

/* The contiguous twin of moe_paged_forward: the same kernels with the page lookup replaced by
 * fixed addressing, for a plan whose pool holds expert e's W1, W3, W2 as pages 3e, 3e+1, 3e+2
 * (shared chunk s as expert E+s).  It exists to measure the cost of the page lookup against
 * a kernel that reads contiguous weights with identical inputs and routing. */
pmoe_status moe_contig_forward(pmoe_plan_t plan, const void* hidden, int32_t T,
                               const float* router_logits, int32_t top_k, void* out,
                               void* workspace, size_t workspace_bytes, pmoe_stream_t stream);

/* The layer forward without any device allocation, for callers that cannot allocate device
 * memory when they run the layer (for example server plugins or embedded runtimes given a fixed
 * device-memory budget at start-up, or latency-critical loops where cudaMalloc would block
 * until in-flight work finishes); they cannot create a plan either, since a plan owns a device
 * allocation.  The paper has no counterpart: this is a convenience of this library.
 * Same arguments and result as moe_paged_forward, with the plan's pool, buffers and descriptor
 * passed directly; it runs the weight-streaming kernels.  Its scratch is one fixed 16 MiB
 * device array inside the library, which every GPU that loads the library holds until the
 * process exits; a call whose layer and T need more returns PMOE_ERR_WORKSPACE (the
 * Qwen1.5-MoE-shaped layer fits up to 16 tokens).  All calls share that array and it keeps the
 * last call's contents, so calls that overlap on the GPU (other streams, other threads) race:
 * serialise them.  device_error (device int32, required: PMOE_ERR_INVALID_ARG when NULL) receives
 * a table error code (an out-of-range page or slot of a routed expert; the output is then
 * undefined) and is not cleared by the call.  The same host checks as pmoe_plan_create apply
 * (descriptor, supported shape, 16-byte aligned pool, load buffers, hidden and out) and run
 * before any device work.  The first call on a device looks up the array's device address
 * (with that device current); make that first call before any stream capture. */
pmoe_status moe_paged_forward_noalloc(const pmoe_layer_desc* desc, const void* page_pool,
                                      int64_t num_pages, const void* load_buf0,
                                      const void* load_buf1, const void* hidden, int32_t T,
                                      const float* router_logits, int32_t top_k,
                                      const int32_t* page_table, const int32_t* buf_slot,
                                      void* out, int32_t* device_error, pmoe_stream_t stream);

/* Double-buffered expert prefetch (Rimuru, section "Expert weights are scattered across
 * pages...": two load buffers alternate, one feeds this layer while the other receives the
 * next layer's experts; section "The adjuster...": finish copying before the table points at
 * the new location).  On copy_stream: wait for `buf_free` (the last reader of buffer `buf` is
 * done; may be NULL), then copy n experts from pinned host memory -- host_experts[i] holds
 * 3*f*d bf16 (W1, W3, W2 back to back) -- into slots slots[i] of load buffer `buf` with one
 * cudaMemcpyAsync each, then record `copy_done` (may be NULL).  n must be <= slots_per_buffer
 * and every slot in [0, slots_per_buffer); host_experts and slots are host arrays. */
pmoe_status pmoe_prefetch_async(pmoe_plan_t plan, int32_t buf, int32_t n,
                                const void* const* host_experts, const int32_t* slots,
                                pmoe_stream_t copy_stream, pmoe_event_t buf_free,
                                pmoe_event_t copy_done);

/* Copy-in of routed experts that are not on the device (Rimuru, section "The pipeline: what
 * happens in one scheduling round": the manager prefetches the experts it predicts a layer needs,
 * the layer's actual routing decides, and an expert the routing picks that is neither cached nor
 * prefetched is copied in before the layer computes).  buf_slot[e] == -2 marks routed expert e as
 * absent: in neither the pool nor a load buffer (a forward call that routes a token to an absent
 * expert sets PMOE_ERR_SLOT_OOB; absent experts no token routes to are never read).  On `stream`,
 * for the T tokens of router_logits (fp32 [T][E], the same top-k rule as the forward): every
 * absent expert some token routes to, in ascending id, takes the next free slot of load buffer
 * `buf` in ascending order (a slot that no buf_slot entry points at), buf_slot[e] (device, updated
 * in place) becomes buf * slots_per_buffer + slot, and its W1 | W3 | W2 are copied from
 * host_experts[e] into the slot.  missed (device int32 [1 + 2E]) receives the count, the experts
 * and their slots: missed[0] = n, missed[1..n] experts, missed[1+E .. 1+E+n) slots.
 *   host_experts  DEVICE array [E] of device-readable pointers (pmoe_device_pointers turns
 *                 pinned host pointers into them), each to 3*f*d bf16 (W1, W3, W2 back to back),
 *                 16-byte aligned; NULL for an expert that has no copy.
 * Run it right before the layer's forward call on the same stream: its kernels let no later
 * kernel start early, so the forward sees the new table entries and the copied bytes.  Nothing
 * else may write load buffer `buf` meanwhile (after a prefetch into it, order the copy-in after
 * that prefetch's copy_done).  Errors in the error word: PMOE_ERR_SLOT_OOB when free slots run
 * out (the experts left over stay absent), PMOE_ERR_INVALID_ARG for an absent routed expert
 * whose host_experts entry is NULL.  Uses plan-owned words, so copy-in and forward calls of one
 * plan must not overlap on the GPU.  T = 0 only sets missed[0] = 0. */
pmoe_status pmoe_copy_in_missing(pmoe_plan_t plan, const float* router_logits, int32_t T,
                                 int32_t* buf_slot, int32_t buf, const void* const* host_experts,
                                 int32_t* missed, pmoe_stream_t stream);

/* The device-side address of each host allocation host[i] (NULL stays NULL), for kernels that
 * read host memory directly (pmoe_copy_in_missing), from cudaHostGetDevicePointer: pinned host
 * memory, and on systems whose GPU reads pageable memory through the host's page tables
 * (Grace-based GB300) pageable memory too.  PMOE_ERR_INVALID_ARG if the runtime gives no device
 * address for one or it is not 16-byte aligned.  Host arrays of n entries. */
pmoe_status pmoe_device_pointers(int32_t n, const void* const* host, void** device);

/* Host-side wait on an event with a timeout (polls cudaEventQuery; never a device spin).
 * PMOE_OK when the event completed, PMOE_ERR_TIMEOUT after timeout_ms milliseconds. */
pmoe_status pmoe_wait_event(pmoe_event_t ev, int32_t timeout_ms);

/* Read (and, if clear != 0, reset to 0) the plan's device error word: 0 or a pmoe_status code
 * raised by a kernel.  Clearing also resets the fused decode path's grid-barrier words.
 * Synchronises with `stream` (NULL = legacy default stream). */
pmoe_status pmoe_get_device_error(pmoe_plan_t plan, int32_t clear, int32_t* code,
                                  pmoe_stream_t stream);

/* ---- single steps, for tests ------------------------------------------------------------ */

/* Top-k softmax routing: logits fp32 [T][E] -> ids int32 [T][k], weights fp32 [T][k]; top-k on
 * the logits with ties to the lower expert id, softmax over all E, optional renormalisation.
 * Device pointers. */
pmoe_status pmoe_route(const float* router_logits, int32_t T, int32_t E, int32_t top_k,
                       int32_t renormalize, int32_t* ids, float* weights, pmoe_stream_t stream);

/* Stable sort-and-pad of the T*(k+S) pairs by expert.  Routed pair i = t*k + j goes to expert
 * ids[i]; shared pair T*k + s*T + t goes to expert E + s.  Experts in ascending id, pairs in
 * ascending index within an expert; an expert with c > 0 pairs owns ceil(c/block_m) blocks,
 * pads hold T*(k+S).  Outputs (device): sorted_ids int32 [>= T*(k+S) + (E+S)*(block_m-1)],
 * block_expert int32 [>= T*(k+S)/block_m + E + S], inv int32 [T*(k+S)] (row of each pair),
 * n_padded int32 [1].  block_m a power of two <= 256; E + S <= 1024.  With scratch != NULL
 * (device, >= pmoe_align_scratch_size() bytes) the sort runs over several CTAs when there are
 * more than 2048 routed pairs (the forward's large-batch form); otherwise in one CTA. */
pmoe_status pmoe_align(const int32_t* ids, int32_t T, int32_t top_k, int32_t E, int32_t S,
                       int32_t block_m, int32_t* sorted_ids, int32_t* block_expert, int32_t* inv,
                       int32_t* n_padded, void* scratch, pmoe_stream_t stream);
size_t pmoe_align_scratch_size(void);

/* Copy experts from pinned host memory straight into pool pages (Rimuru, section "The
 * adjuster...": an expert the adjuster adds is written into the pages it reserved for it, and
 * the page table points at them only after the copy).  On copy_stream: wait for `after` (e.g.
 * the end of the forward pass that last read those pages; may be NULL), then for each expert i
 * copy matrix j (W1, W3, W2) of host_experts[i] (3*f*d bf16, back to back) into pool page
 * pages[3*i + j] with one cudaMemcpyAsync each, then record `copy_done` (may be NULL).  pages is
 * a host int32 array [n][3] of distinct pages in [0, num_pages) (PMOE_ERR_PAGE_OOB otherwise). */
pmoe_status pmoe_fill_pages_async(pmoe_plan_t plan, int32_t n, const void* const* host_experts,
                                  const int32_t* pages, pmoe_stream_t copy_stream,
                                  pmoe_event_t after, pmoe_event_t copy_done);

/* ---- remapped contiguous view (the rival design to the page lookup) --------------------------
 *
 * FluxMoE (awesome-system-papers, section "核心方法", PagedTensor): instead of looking pages up
 * inside the kernel, keep a stable virtual address range per logical weight tensor and map
 * physical blocks under it with the CUDA driver's virtual memory calls before the kernel runs,
 * so an unmodified contiguous kernel reads scattered physical memory.  Invariants it states:
 * stable virtual addresses; a virtual page maps at most one physical block at a time; a block is
 * reused only after every kernel reading it has finished; the blocks form a fixed pool.
 *
 * Here one block is one expert page (f*d bf16), which must be a multiple of the device's VMM
 * granularity (pmoe_vmm_granularity; 2 MiB pages for d=2048, f=512 or d=4096, f=14336, not for
 * d=2048, f=1408).  pmoe_vmm_create allocates n_blocks physical blocks and reserves two device
 * address ranges: `blocks` maps block i at offset i*block_bytes (all blocks, for the page-table
 * forward) and `view` holds n_virtual virtual pages, unmapped at first (for moe_contig_forward,
 * expert e's matrix j at virtual page 3e+j).  Both ranges alias the same physical bytes: no
 * copy.  Reading an unmapped virtual page faults the GPU, so a caller launches a kernel on the
 * view only once every page that kernel can read is mapped (pmoe_vmm_lookup).  All calls are
 * host calls; they allocate device memory only in pmoe_vmm_create and free it in
 * pmoe_vmm_destroy, and each makes the view's device current for its driver calls and then puts
 * the caller's current device back.  Driver failures return PMOE_ERR_CUDA with
 * pmoe_last_error() set. */
typedef struct pmoe_vmm* pmoe_vmm_t;

/* Smallest block size (bytes) the device's VMM maps, or 0 with a status on error. */
pmoe_status pmoe_vmm_granularity(int32_t device, size_t* bytes);
pmoe_status pmoe_vmm_create(int32_t device, size_t block_bytes, int64_t n_blocks, int64_t n_virtual,
                            pmoe_vmm_t* out);
pmoe_status pmoe_vmm_destroy(pmoe_vmm_t vmm);
/* Device pointers of the two ranges (either may be NULL). */
pmoe_status pmoe_vmm_pointers(pmoe_vmm_t vmm, void** blocks, void** view);
/* Map block blocks[i] under virtual page virt[i] for i < n (PMOE_ERR_INVALID_ARG, nothing
 * mapped, if a virtual page is already mapped, listed twice or out of range). */
pmoe_status pmoe_vmm_map(pmoe_vmm_t vmm, int64_t n, const int64_t* virt, const int64_t* blocks);
/* Unmap virtual pages virt[i] once `readers_done` (the last kernel reading them; may be NULL)
 * has completed, waiting on the host for at most timeout_ms (PMOE_ERR_TIMEOUT, nothing unmapped). */
pmoe_status pmoe_vmm_unmap(pmoe_vmm_t vmm, int64_t n, const int64_t* virt,
                           pmoe_event_t readers_done, int32_t timeout_ms);
/* The block under each virtual page (-1: unmapped), host int64 [n_virtual]. */
pmoe_status pmoe_vmm_lookup(pmoe_vmm_t vmm, int64_t* block_of);

/* ---- exponent-only Huffman compression of bf16 expert pages ----------------------------------
 *
 * FluxMoE (awesome-system-papers, section "核心方法", observation 3 and the compressed GPU
 * backend): bf16 expert weights keep sign and mantissa as they are and Huffman-code the 8-bit
 * exponent, whose entropy is low; the GPU decompresses before the weights are read.  Format (the
 * page fixes none): per page of n values, code lengths [256], n, stream bits, a 4096-entry decode
 * table (symbol | length << 8 for the next 12 stream bits), the start bit of each chunk of at
 * most 256 values (within each group of 65536 values, runs of 8 values are dealt to the group's
 * chunks in turn, so the threads decoding neighbouring chunks read and write neighbouring runs),
 * the sign|mantissa bytes in value order and the exponent stream (32-bit words, bit 31 first,
 * two zero words after it); sections 16-byte aligned.  Codes are canonical Huffman codes of at most 12 bits.
 * Lossless: decoding gives back every bit pattern (NaN, infinities, subnormals included). */

/* Bytes pmoe_exp_encode may write for n values. */
size_t pmoe_exp_encode_bound(int64_t n);
/* Host encoder: values (host bf16 bit patterns) -> out (host, cap >= pmoe_exp_encode_bound(n));
 * *bytes = the blob's size.  n * 12 must stay below 2^32. */
pmoe_status pmoe_exp_encode(const uint16_t* values, int64_t n, void* out, size_t cap, size_t* bytes);
/* GPU decoder: decode n_pages blobs (device, 16-byte aligned, src_bytes[i] bytes each, every one of
 * n values) into dst[i] (device, 16-byte aligned, n bf16) on `stream`, one thread per 256 values.
 * src, src_bytes and dst are host arrays, n_pages <= 128.  A blob whose header does not match n or
 * its size sets *device_error (device int32, may be NULL) to PMOE_ERR_INVALID_ARG and leaves its
 * chunks unwritten. */
pmoe_status pmoe_exp_decode_async(int32_t n_pages, int64_t n, const void* const* src,
                                  const int64_t* src_bytes, void* const* dst, int32_t* device_error,
                                  pmoe_stream_t stream);

/* ---- three tiers of pages over one pool -----------------------------------------------------
 *
 * Rimuru, section "One pool for data whose sizes differ by orders of magnitude": the pool is one
 * byte range read through views with different page sizes.  Huge pages (size lcm(expert page,
 * SSM page), or the expert page without SSM state) split on demand into middle pages (expert or
 * SSM pages, one kind per huge page); an expert page splits into small pages (KV cache or
 * convolution-state pages, one kind per split page).  A small page comes from, in order: a free
 * small page of the same kind in a split page that already holds a live page of the same owner
 * (the request: pages of one request are freed together), any free small page of that kind, a
 * free expert page split for it, a free huge page split into expert pages first.  A huge page is
 * never cut straight into small pages.  A middle page comes from a free page of its kind, else a
 * split huge page.  Ties go to the lowest byte offset.  Freeing runs upward: a split expert page
 * whose small pages are all free is an expert page again, and a huge page whose middle pages are
 * all free returns to the huge pages.
 *
 * Sizes in bytes: expert_page > 0; ssm_page >= 0 (0: none); kv_page and conv_page (0: none) must
 * divide expert_page.  pool_bytes / huge page is the number of huge pages (the rest is unused).
 * Offsets are byte offsets into the pool; an expert page at offset o is page o / expert_page of
 * the kernels' page pool.  Host only; the caller owns the pool memory. */
typedef struct pmoe_tiers* pmoe_tiers_t;
enum { PMOE_PAGE_EXPERT = 0, PMOE_PAGE_SSM = 1, PMOE_PAGE_KV = 2, PMOE_PAGE_CONV = 3 };

pmoe_status pmoe_tiers_create(int64_t pool_bytes, int64_t expert_page, int64_t ssm_page,
                              int64_t kv_page, int64_t conv_page, pmoe_tiers_t* out);
pmoe_status pmoe_tiers_destroy(pmoe_tiers_t t);
/* One page of `kind` for `owner` (owner matters for small pages only): *offset = its byte offset,
 * or -1 when the pool has no room (not an error). */
pmoe_status pmoe_tiers_alloc(pmoe_tiers_t t, int32_t kind, int64_t owner, int64_t* offset);
/* Return a live page (PMOE_ERR_INVALID_ARG, nothing changed, if `offset` is not a live page of
 * `kind`). */
pmoe_status pmoe_tiers_free(pmoe_tiers_t t, int32_t kind, int64_t offset);
/* counts[8]: huge page bytes, free huge pages, free expert pages, free SSM pages, live expert
 * pages, live SSM pages, split expert pages, free small pages (KV + conv). */
pmoe_status pmoe_tiers_stats(pmoe_tiers_t t, int64_t* counts);

/* ---- the adjuster: which experts each layer keeps in the page pool -------------------------
 *
 * Host only (no device work).  Rimuru, section "The adjuster: when to evict an expert, and which
 * one?": after the scheduler has placed the round's requests it is short of
 * R_b expert pages or has F_b free ones, and the adjuster
 *   - evicts ceil((R_b + 1) / 3) experts when R_b > 0,
 *   - else evicts 1 expert when F_b < 2,
 *   - else adds min(5, floor((F_b - 9) / 3)) experts when F_b > 9 (nothing for 2 <= F_b <= 9).
 * Every expert takes 3 pages (W1, W3, W2).  Each layer keeps the top slice of an offline ranking
 * of its experts by routing probability (probs[l][e], ties to the lower expert id).  To add,
 * each layer with an uncached expert nominates the next one of its ranking and the adjuster
 * takes the nominees with the highest probability; to evict, each layer that keeps an expert and
 * offloads fewer than offload_limit nominates the last expert it keeps and the adjuster takes
 * the nominees with the lowest probability; at most one per layer per round (ties to the lower
 * layer).  An added expert gets 3 free pages at once (lowest page ids first: the reserved pages
 * it is copied into before the page table points at them).  An evicted expert's pages stay its
 * own until pmoe_adjuster_end_forward (the forward pass running now may still read them), then
 * return to the free pages.  F_b counts free pages only; pages lent out (KV cache pages of the
 * unified pool) are neither free nor an expert's.  Errors: argument checks return
 * PMOE_ERR_INVALID_ARG with pmoe_last_error() set and leave the state unchanged; no call blocks
 * or touches a device.  One adjuster must not be used from two threads at once. */
typedef struct pmoe_adjuster* pmoe_adjuster_t;

/* probs: host fp32 [n_layers][n_experts] routing probabilities (finite); cached: host int32
 * [n_layers], how many top-ranked experts each layer keeps at the start (0..n_experts); they
 * take pages 0, 1, 2, ... layer by layer in ranking order (W1, W3, W2 of each expert), the rest
 * of the num_pages pages are free.  num_pages >= 3 * sum(cached), < 2^31.  offload_limit >= 0:
 * a layer with n_experts - kept >= offload_limit is left out of shrinking.  The adjuster copies
 * what it needs; the caller keeps ownership of probs and cached and destroys *out. */
pmoe_status pmoe_adjuster_create(int32_t n_layers, int32_t n_experts, const float* probs,
                                 int32_t offload_limit, const int32_t* cached, int64_t num_pages,
                                 pmoe_adjuster_t* out);
pmoe_status pmoe_adjuster_destroy(pmoe_adjuster_t adj);

/* One round.  short_pages = R_b (>= 0).  Writes records of 6 int32 to changes (host):
 * {+1 add / -1 evict, layer, expert, page of W1, page of W3, page of W2}, in the order taken
 * (a round only adds or only evicts); *n_changes = the records written.  A round takes no more
 * than max_changes (>= 0) changes, nor more than one per layer.  PMOE_ERR_INVALID_ARG while the
 * evictions of the previous round still wait for pmoe_adjuster_end_forward. */
pmoe_status pmoe_adjuster_decide(pmoe_adjuster_t adj, int32_t short_pages, int32_t max_changes,
                                 int32_t* changes, int32_t* n_changes);

/* The forward pass that ran during the round has ended: evicted experts' pages become free. */
pmoe_status pmoe_adjuster_end_forward(pmoe_adjuster_t adj);

/* Lend n free pages (lowest ids first) to the caller, e.g. for KV cache (PMOE_ERR_INVALID_ARG
 * when fewer than n are free), and take lent pages back. */
pmoe_status pmoe_adjuster_lend(pmoe_adjuster_t adj, int32_t n, int32_t* pages);
pmoe_status pmoe_adjuster_give_back(pmoe_adjuster_t adj, int32_t n, const int32_t* pages);

/* State: free pages (F_b), the experts each layer keeps (cached int32 [n_layers], may be NULL),
 * and a layer's page table (int32 [n_experts][3]; -1 for an expert not kept, an evicted expert
 * keeps its pages until pmoe_adjuster_end_forward). */
pmoe_status pmoe_adjuster_state(pmoe_adjuster_t adj, int64_t* free_pages, int32_t* cached);
pmoe_status pmoe_adjuster_page_table(pmoe_adjuster_t adj, int32_t layer, int32_t* page_table);

#ifdef __cplusplus
}
#endif

#endif /* PMOE_H */
