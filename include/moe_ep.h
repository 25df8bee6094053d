/*
 * moe_ep.h -- C ABI of libmoe_ep.so: MoE token dispatch / combine on one GPU.
 *
 * The operators are the dispatch and combine of expert-parallel MoE layers
 * as Hybrid-EP and DeepEP implement them: dispatch sends every token to the
 * ranks that hold its top-K experts, combine brings the expert outputs back
 * to the token's original position ("Inside the Nebius + PyTorch DeepSeek V3
 * recipe", section "Mixture-of-experts and wide expert parallelism";
 * Hybrid-EP news article, section "Technical Structure").  Here the EP ranks
 * are virtual: contiguous blocks of E/R experts whose receive rows live in
 * one packed buffer in this GPU's HBM, so there is no cross-GPU transport.
 *
 * Conventions shared by every call:
 *  - All tensors are row-major device memory owned by the caller.  The
 *    library allocates nothing and never synchronises inside the three
 *    operator calls (moe_dispatch_layout, moe_dispatch, moe_combine).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Work is enqueued in stream order and the call returns at once.
 *  - Host-side argument checks return a moe_status synchronously and enqueue
 *    nothing on failure.  A failed kernel launch returns MOE_ERR_CUDA.
 *  - Device-side problems (an expert id outside [-1, E), a slot outside the
 *    buffers, a bounded wait that ran out) never fault: the offending access
 *    is skipped, a bit is set in the layout's device status word and the
 *    kernel goes on or returns.  moe_layout_read_status() reports it.
 *  - bf16 is passed as uint16_t bit patterns; FP8 is OCP E4M3 bytes.
 *  - Calls that share one moe_layout must be stream-ordered (one stream, or
 *    events between streams); overlapping calls on one layout race.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer        */
    MOE_ERR_CAPACITY = 2,      /* device: a slot fell outside the buffers     */
    MOE_ERR_TIMEOUT = 3,       /* device: a bounded wait ran out              */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed        */
    MOE_ERR_UNSUPPORTED = 5,   /* sizes beyond the documented limits          */
    MOE_ERR_EXPERT_ID = 6      /* device: an expert id outside [-1, E)        */
} moe_status;

/* Bits of the device status word (moe_layout.status). */
#define MOE_DEVERR_EXPERT_ID 0x1u
#define MOE_DEVERR_CAPACITY  0x2u
#define MOE_DEVERR_TIMEOUT   0x4u

/* Limits (MOE_ERR_UNSUPPORTED beyond them). */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK    32
#define MOE_MAX_RANKS   256

/* Test hook bits for moe_tuning.debug_flags (0 in production). */
#define MOE_DEBUG_STALL_FIRST_TILE 0x1u  /* layout: the first scan tile never publishes,
                                            so its successors' bounded waits run out */

/* Optional launch tuning; pass NULL for the defaults. */
typedef struct moe_tuning {
    int32_t  num_channels;     /* CTAs ("independent channels") for dispatch / combine; 0 = auto
                                  (dispatch: one item per warp (32-byte kernel) or per CTA
                                  (TMA kernel); 16-byte vector dispatch and combine: four waves
                                  of resident CTAs)                                              */
    int32_t  stages;           /* dispatch pipeline depth per channel, 2..8; 0 = auto (TMA
                                  kernels: at most the items a channel holds; variant 2: 2 / 4 / 8
                                  = batches of 1 / 2 / 4 items, two batches in flight)          */
    int32_t  chunk_bytes;      /* dispatch: bf16 bytes of a row per pipeline item (a multiple of
                                  256, >= 256); 0 = 16384, i.e. whole rows up to hidden 8192     */
    int32_t  variant;          /* dispatch / combine kernel: 0 = default (dispatch: 4, or where
                                  its alignment does not hold, 1 for bf16 and 2 for FP8 /
                                  MXFP8; combine: 16-byte vector loads with the fma chain in
                                  registers), 1 = TMA bulk copies staged in
                                  shared memory (combine: K <= 8), 2 = 16-byte vector loads /
                                  stores (combine: as 0), 3 = FP8 / MXFP8 dispatch with
                                  warp-specialised roles (one TMA warp, eight quantiser warps;
                                  bf16 dispatch and combine treat 3 as 0), 4 = dispatch with
                                  32-byte vector loads / stores, a lane per 32 columns (needs
                                  x and recv_x 32-byte aligned and, for bf16, hidden % 16 == 0;
                                  otherwise it runs as 1 for bf16 and as 2 for FP8 / MXFP8;
                                  combine: the 32-byte gather, one warp per 512-column segment,
                                  with the same alignment rule, else as 0)                       */
    uint64_t wait_timeout_ns;  /* bound on every device-side wait; 0 = 1 second                   */
    uint32_t debug_flags;      /* MOE_DEBUG_* test hooks                                          */
    uint32_t reserved2;
} moe_tuning;

/*
 * Routing layout.  Notation: T tokens, K top-k, E experts, R virtual ranks,
 * m = E / R experts per rank, rank(e) = e / m (contiguous expert blocks;
 * the pages say each GPU holds a subset, e.g. 8 of 256 experts, but not
 * which one).
 *
 *  tokens_per_expert[E]    #{(t,k) : topk_idx[t,k] == e}
 *  expert_offset[E+1]      exclusive prefix of tokens_per_expert
 *  tokens_per_rank[R]      #{t : token t has an expert on rank r}
 *  rank_offset[R+1]        first receive row of each rank; rank_offset[R] = number of pairs
 *  recv_expert_offset[E+1] exclusive prefix of the per-expert counts of
 *                          "primary" pairs: the primary expert of (t, r) is
 *                          the smallest id token t has on rank r
 *  recv_slot[T,R]          receive row of token t on rank r, or -1.  Rows are
 *                          ordered by (primary expert, token), so each rank's
 *                          rows are contiguous and grouped by expert.
 *  expert_slot[T,K]        expert-major row of entry (t,k), ordered by
 *                          (expert, token, k); -1 for a masked entry
 *  recv_src_token[cap]     token of each receive row; -1 past the last pair
 *  expert_src_row[T*K]     receive row holding each expert-major row's token; -1 past the end
 *  expert_weight[T*K]      router weight of each expert-major row; 0 past the end
 *  status                  device status word (MOE_DEVERR_* bits) of the latest
 *                          moe_dispatch_layout and the calls after it
 *
 * The receive buffer is preallocated for the worst case, capacity >=
 * T * min(K, R) rows (Hybrid-EP news article, "Availability and
 * Integration": worst-case buffer preallocation for dynamic routing), so no
 * count has to travel back to the host.
 */
typedef struct moe_layout {
    int32_t T, K, E, R;
    int64_t capacity;
    int32_t tile_tokens;        /* tokens per scan tile, fixed at init */
    int32_t num_tiles;
    int32_t num_sources;        /* 0: the single-source layout above; S >= 1: the
                                   multi-source receive layout (below)          */
    int32_t source_tokens;      /* tokens per source, T / S (T when num_sources == 0) */
    int32_t *tokens_per_expert, *expert_offset, *tokens_per_rank, *rank_offset;
    int32_t *recv_expert_offset, *recv_slot, *expert_slot, *recv_src_token, *expert_src_row;
    float   *expert_weight;
    int32_t *recv_source_offset; /* [R, S+1], multi-source layout only; NULL otherwise */
    uint32_t *status;
    void    *workspace;         /* scan scratch, carved from the same memory */
    size_t   workspace_bytes;
} moe_layout;

/* Bytes of device memory moe_layout_init needs for these sizes (outputs +
 * scan workspace, each array 256-byte aligned).  0 if the sizes are invalid.
 * This is the layout's workspace-size query; it takes the capacity as well
 * as T, K, E and R because one of the outputs it sizes, recv_src_token, has
 * one entry per receive row. */
size_t moe_layout_bytes(int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity);

/* Carve the layout's arrays out of caller memory.  Host only: no CUDA call.
 * `device_mem` must be 256-byte aligned, hold moe_layout_bytes(...) bytes and
 * be ZERO-FILLED before its first use (the scan's progress flags start at
 * zero); afterwards the library keeps it consistent itself.
 * capacity must be >= T * min(K, R). */
moe_status moe_layout_init(moe_layout* L, int32_t T, int32_t K, int32_t E, int32_t R,
                           int64_t capacity, void* device_mem, size_t bytes);

/*
 * Multi-source receive layout: the single-GPU stand-in for the exchange in
 * which every source rank sends its tokens to the ranks of their experts and
 * every destination rank receives from all sources ("Inside the Nebius +
 * PyTorch DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
 * parallelism").  S sources of Ts tokens each; token g of the concatenated
 * routing topk_idx [T, K], T = S * Ts, belongs to source g / Ts.  Destination
 * r owns its own receive region, rows [r*T, (r+1)*T) -- its worst case, every
 * token of every source -- so capacity = R * T.  The tokens that reach r fill
 * the region from its start in (source, token) order, i.e. ascending g.
 *
 *  recv_slot[T,R]           r*T + #{g' < g : g' has a valid expert on r}, or -1
 *  tokens_per_rank[R]       rows used in region r
 *  rank_offset[R+1]         r*T, the region starts; rank_offset[R] = R*T
 *  recv_source_offset[R,S+1] #{g < s*Ts : g reaches r}: source s's rows in
 *                           region r are [off[r,s], off[r,s+1]) counted from
 *                           the region start; off[r,S] = tokens_per_rank[r]
 *  recv_src_token[R*T]      g of each used row; -1 in the unused tail of every region
 *  recv_expert_offset       NULL: the rows are not grouped by expert
 *
 * The expert-major outputs (tokens_per_expert, expert_offset, expert_slot,
 * expert_src_row, expert_weight) are those of the single-source layout over
 * all T tokens.  moe_dispatch, moe_combine, moe_dispatch_backward and
 * moe_combine_backward take either kind of layout unchanged; the layout call
 * adds a third kernel that reads the per-source offsets off the sorted
 * regions.
 */
#define MOE_MAX_SOURCES 1024

/* Bytes for moe_layout_init_sources; 0 if the sizes are invalid. */
size_t moe_layout_sources_bytes(int32_t S, int32_t source_tokens, int32_t K, int32_t E, int32_t R);

/* As moe_layout_init, for the multi-source layout (capacity R * S * Ts).
 * 1 <= S <= MOE_MAX_SOURCES and R * S * Ts must fit in int32. */
moe_status moe_layout_init_sources(moe_layout* L, int32_t S, int32_t source_tokens, int32_t K, int32_t E,
                                   int32_t R, void* device_mem, size_t bytes);

/* Dispatch layout: counts, prefix offsets and token<->slot maps (all fields
 * above), which size and address the worst-case-preallocated receive buffer
 * (Hybrid-EP news article, "Availability and Integration"; the token-to-rank
 * routing of "Inside the Nebius + PyTorch DeepSeek V3 recipe", "Mixture-of-
 * experts and wide expert parallelism").  Inputs: topk_idx int32 [T,K]
 * (-1 = masked) and topk_w fp32 [T,K] (may be NULL: expert_weight is then
 * zero-filled).  Two kernels: a warp-aggregated per-tile histogram with a
 * decoupled-lookback scan over E-wide count vectors (up to one tile per SM,
 * the tile is the block index and all tiles are resident at once; more tiles
 * claim ids from a ticket so every wait is on a running CTA; every wait is
 * bounded), then a finalize pass.
 * num_experts / num_ranks must equal L->E / L->R. */
moe_status moe_dispatch_layout(const int32_t* topk_idx, const float* topk_w,
                               int32_t num_experts, int32_t num_ranks,
                               moe_layout* L, void* stream, const moe_tuning* tuning);

/* Dispatch layout for callers that cannot allocate device memory.
 *
 * Some callers of this library never call cudaMalloc themselves: a plugin
 * inside a host framework that hands out every device buffer from its own
 * allocator and refuses side allocations, or a serving loop that has fixed
 * its device memory at start-up and must not pay an allocation's latency and
 * implicit device synchronisation on the request path.  Such a caller can
 * still own the layout's outputs (they are what it keeps), but not the scan's
 * scratch space.  This entry point has no counterpart on the pages: it is the
 * same operation as moe_dispatch_layout, with identical results, and it
 * allocates nothing.
 *
 * The scan workspace is a device array of MOE_NOALLOC_SCRATCH_BYTES compiled
 * into the library; every GPU that loads the library holds it until the
 * process exits.  Sizes whose workspace does not fit (moe_layout_bytes minus
 * the outputs; about 8 * T * K bytes plus 16 * E to 32 * E bytes per
 * 2048-entry tile) return MOE_ERR_UNSUPPORTED.
 *
 * Fields of *L that are read: T, K, E, R, capacity (>= T * min(K, R)), the
 * ten output pointers and status, all caller-owned device memory of the sizes
 * listed above; tile_tokens, num_tiles, workspace and workspace_bytes are
 * ignored and left unchanged.  No moe_layout_init call is needed.  For the
 * multi-source layout also num_sources and source_tokens (T = S * Ts,
 * capacity = R * T) and recv_source_offset instead of recv_expert_offset.
 *
 * All calls share the one array, which keeps the previous call's contents;
 * each call clears the parts that must start at zero.  Calls that overlap on
 * the GPU (on different streams without ordering, or from several threads)
 * race on it.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it, keyed by the
 * device's current context: make that first call before any stream capture.
 * After a cudaDeviceReset the next call looks the address up again in the new
 * context (also before any capture).  No cudaMalloc, cudaFree or other
 * allocating routine is called. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)

moe_status moe_dispatch_layout_noalloc(const int32_t* topk_idx, const float* topk_w,
                                       int32_t num_experts, int32_t num_ranks,
                                       moe_layout* L, void* stream, const moe_tuning* tuning);

/* Receive formats of moe_dispatch. */
#define MOE_FORMAT_BF16  0   /* bf16 rows                                              */
#define MOE_FORMAT_FP8   1   /* E4M3 rows + one fp32 scale per 1x128 block             */
#define MOE_FORMAT_MXFP8 2   /* E4M3 rows + one E8M0 byte per 1x32 block (OCP MX)      */

/* Dispatch: for every pair with recv_slot[t,r] >= 0 write token t's row into
 * receive row recv_slot[t,r]: each token once per destination rank, rows in
 * expert-contiguous order.
 *   MOE_FORMAT_BF16: recv_x is bf16 [capacity, hidden]; recv_scales must be NULL.
 *   MOE_FORMAT_FP8: recv_x is E4M3 bytes [capacity, hidden] and recv_scales
 *     fp32 [capacity, hidden/128]: per token and 1x128 block, s = amax / 448
 *     (fp32, round to nearest), q = E4M3(x / s) with round-to-nearest-even and
 *     saturation; an all-zero block gives s = 0 and q = 0.  FP8 dispatch:
 *     "MoE / Hybrid-EP Validation", "FP8 dispatch restriction"; the pages give
 *     no recipe, this one is the DeepEP-style 1x128 block scaling.
 *   MOE_FORMAT_MXFP8: recv_x is E4M3 bytes [capacity, hidden] and recv_scales
 *     E8M0 bytes [capacity, hidden/32] (OCP Microscaling MXFP8, the format of
 *     the MXFP8 training on the Hybrid-EP news article, "Efficiency
 *     Numbers"): per 1x32 block se = floor(log2(amax)) - 8 clamped to
 *     [-127, 127] (-127 for an all-zero block), byte = se + 127,
 *     q = E4M3(x * 2^-se), round to nearest even, saturating at 448.
 * x is bf16 [T, hidden]; hidden % 8 == 0 (hidden % 128 == 0 for both FP8
 * formats); x, recv_x 16-byte aligned, recv_scales 4-byte aligned.  Rows
 * past rank_offset[R] are not written.  Default kernel (every format, when x
 * and recv_x are 32-byte aligned): each warp moves one 1024-column segment of
 * one token -- two 32-byte loads per lane, the FP8 / MXFP8 codes computed in
 * registers -- and writes it with one 32-byte store per lane to every
 * destination row; no grid-wide synchronisation.  16-byte aligned calls take
 * the staged kernel for bf16 (each CTA an independent channel: TMA bulk loads
 * of a row chunk into shared memory, then one TMA bulk store per destination
 * row; Hybrid-EP news article, "Technical Structure") and the 16-byte vector
 * kernel for FP8 / MXFP8. */
moe_status moe_dispatch(const uint16_t* x, int32_t hidden, const moe_layout* L, int32_t format,
                        void* recv_x, void* recv_scales, void* stream, const moe_tuning* tuning);

/* moe_dispatch_layout followed by moe_dispatch, in one call: the same
 * arguments and checks as the two calls, the same results in L, recv_x and
 * recv_scales (the dispatch uses num_experts, num_ranks and L exactly as the
 * layout call leaves them).  Dispatch sends each token to the ranks its
 * layout assigns ("Inside the Nebius + PyTorch DeepSeek V3 recipe",
 * "Mixture-of-experts and wide expert parallelism"), so the two always come
 * in this order.  Because x is an input of this one call -- complete before
 * its first kernel starts, like topk_idx -- the dispatch may read x while the
 * layout is still being computed: for bf16 and MXFP8 rows the default kernel
 * becomes resident while the layout runs, and each warp loads (MXFP8: and
 * quantises) its segment of x before it waits for the slots.  With two
 * separate calls the dispatch cannot, since the caller may write x between
 * them.  FP8 rows (no gain measured) run as the two calls do.  tuning
 * applies to both parts as in the two calls. */
moe_status moe_dispatch_with_layout(const int32_t* topk_idx, const float* topk_w, int32_t num_experts,
                                    int32_t num_ranks, moe_layout* L, const uint16_t* x, int32_t hidden,
                                    int32_t format, void* recv_x, void* recv_scales, void* stream,
                                    const moe_tuning* tuning);

/* Combine: the expert outputs back to each token's position, weighted by the
 * router ("Inside the Nebius + PyTorch DeepSeek V3 recipe", "Mixture-of-
 * experts and wide expert parallelism"; Hybrid-EP news article, "Technical
 * Structure"):
 * out[t,:] = bf16_rne( sum over k = 0..K-1 with expert_slot[t,k] >= 0
 * of topk_w[t,k] * y[expert_slot[t,k], :] ), accumulated in fp32 as a fused
 * multiply-add chain starting from 0 in ascending k.  y is bf16 [T*K, hidden]
 * in expert-major row order (row expert_offset[e] + j is expert e's j-th
 * entry); out is bf16 [T, hidden]; a token with every entry masked gets +0.
 * hidden % 8 == 0; y and out 16-byte aligned.  moe_tuning.variant 4 takes the
 * 32-byte gather (one warp per 512-column segment of a token, the valid
 * slots found by one ballot; needs y and out 32-byte aligned and hidden % 16
 * == 0, else it runs as 0).  Every variant gives the same bits; the default
 * measured fastest for the combine's dense rows. */
moe_status moe_combine(const uint16_t* y, int32_t hidden, const moe_layout* L,
                       const float* topk_w, uint16_t* out, void* stream, const moe_tuning* tuning);

/* Low-latency (decode) dispatch into a fixed-capacity per-expert buffer.
 * DeepEP pairs its high-throughput kernels with low-latency ones for decode
 * ("Inside the Nebius + PyTorch DeepSeek V3 recipe", section "DeepEP"); their
 * receive buffer has a static shape so the experts run on fixed-size inputs.
 * Here every valid entry (t,k) of expert e = topk_idx[t,k] is written to row
 * e * cap_per_expert + j of recv bf16 [E, cap_per_expert, hidden], j = the
 * entry's position among e's entries in (t,k) order (each token once per
 * expert, not per rank).  Entries with j >= cap_per_expert are dropped
 * (ll_slot -1, MOE_DEVERR_CAPACITY).  Outputs: tokens_per_expert[E] = rows
 * written, ll_slot int32 [T,K] = row or -1, and the device status word
 * *status (MOE_DEVERR_* bits, overwritten by this call).  One launch, no
 * workspace: T * K <= 4096 (MOE_ERR_UNSUPPORTED beyond).  Rows of recv that
 * receive nothing are not written. */
moe_status moe_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E, int32_t hidden,
                           int32_t cap_per_expert, uint16_t* recv, int32_t* tokens_per_expert, int32_t* ll_slot,
                           uint32_t* status, void* stream, const moe_tuning* tuning);

/* Combine over the low-latency layout: out[t,:] = bf16_rne(fp32 fused
 * multiply-add chain over k ascending of topk_w[t,k] * y[ll_slot[t,k], :]),
 * skipping ll_slot < 0; y is bf16 [E, cap_per_expert, hidden].  Slots past the
 * buffer set MOE_DEVERR_CAPACITY in *status (OR-ed in) and are skipped. */
moe_status moe_ll_combine(const uint16_t* y, const int32_t* ll_slot, const float* topk_w, int32_t T, int32_t K,
                          int32_t E, int32_t hidden, int32_t cap_per_expert, uint16_t* out, uint32_t* status,
                          void* stream, const moe_tuning* tuning);

/* Backward of the bf16 dispatch (its adjoint): grad_x[t,:] = bf16_rne(sum over
 * r = 0..R-1 with recv_slot[t,r] >= 0 of grad_recv[recv_slot[t,r], :]),
 * accumulated in fp32 in ascending r (0 for a token sent nowhere).
 * grad_recv is bf16 [capacity, hidden] (the gradient of the receive rows);
 * grad_x is bf16 [T, hidden].  hidden % 8 == 0, 16-byte aligned rows.  With
 * grad_recv and grad_x 32-byte aligned and hidden % 16 == 0 it runs the
 * 32-byte gather of moe_combine's variant 4: each token's valid ranks come
 * from one ballot over its recv_slot row; otherwise the 16-byte gather of
 * moe_combine.  Both give the same bits.
 * Training is the pages' workload (Hybrid-EP news article, "Efficiency
 * Numbers"); they do not describe the backward pass: this is the adjoint of
 * the forward definition. */
moe_status moe_dispatch_backward(const uint16_t* grad_recv, int32_t hidden, const moe_layout* L,
                                 uint16_t* grad_x, void* stream, const moe_tuning* tuning);

/* Backward of moe_combine, from grad_out bf16 [T, hidden]:
 *   grad_y[expert_slot[t,k], :] = bf16_rne(fp32(topk_w[t,k] * grad_out[t, :]))
 *   grad_w[t,k] = sum_h grad_out[t,h] * y[expert_slot[t,k], h]   (fp32; 0 if masked)
 * y and grad_y are bf16 [T*K, hidden] in expert-major row order (rows no
 * entry maps to are not written); grad_w is fp32 [T, K].  The dot products are
 * fp32 fused multiply-adds reduced in a fixed order (deterministic), one CTA
 * per token; their rounding differs from an exact sum by at most about
 * hidden * 2^-24 * sum_h |grad_out * y|. */
moe_status moe_combine_backward(const uint16_t* grad_out, const uint16_t* y, int32_t hidden, const moe_layout* L,
                                const float* topk_w, uint16_t* grad_y, float* grad_w, void* stream,
                                const moe_tuning* tuning);

/* Helpers of this library (the pages define no error interface; these two
 * only read back and name the status of the calls above). */

/* Synchronise `stream`, read the device status word, and map it to a status
 * (timeout first -- a timed-out scan also makes later kernels see slots out
 * of range -- then expert ids, then capacity).  `flags_out` (may be NULL)
 * receives the raw MOE_DEVERR_* bits. */
moe_status moe_layout_read_status(const moe_layout* L, void* stream, uint32_t* flags_out);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status s);

/* Number of SMs of the current device (0 on error); used for channel counts. */
int32_t moe_device_sm_count(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_EP_H */
