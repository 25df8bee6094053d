/*
 * moe_oracle.h -- plain single-threaded CPU oracle for MoE token dispatch / combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this code; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code with the CUDA
 * library (include/moe_ep.h) and neither side includes the other.
 *
 * What is computed (sources: "Inside the Nebius + PyTorch DeepSeek V3 recipe",
 * section "Mixture-of-experts and wide expert parallelism": dispatch sends each
 * token to its top-K experts, which are partitioned across EP ranks, combine
 * returns the expert outputs to the tokens' original positions; Hybrid-EP
 * news article (cryptojournalpost, Feb 2 2026), sections "Technical
 * Structure" and "Availability and Integration": dispatch and combine
 * operators, worst-case preallocated receive buffers; "MoE / Hybrid-EP
 * Validation", section "FP8 dispatch restriction": dispatch may carry FP8).
 * The pages give no layout, ordering or quantisation formula; the readings
 * used here are:
 *
 *   - experts are split into R contiguous blocks of m = E/R; rank(e) = e / m;
 *   - a token is sent once per destination rank; within the packed receive
 *     buffer rows are ordered by (primary expert, token), the primary expert
 *     of (t, r) being the smallest expert id of token t that lives on rank r;
 *   - expert-major rows (the y layout) are ordered by (expert, t, k);
 *   - FP8 is OCP E4M3 (bias 7, max 448, no inf) with one fp32 scale per
 *     1x128 block: s = amax / 448 (fp32 RN), q = e4m3_rne_satfinite(x / s);
 *     an all-zero block gives s = 0 and q = 0x00;
 *   - combine: acc = 0; for k ascending, acc = fma(w[t,k], y, acc) in fp32;
 *     out = bf16_rne(acc).
 *
 * Every array is host memory, row-major, owned by the caller.  Return value:
 * 0 on success, otherwise a bitwise OR of MOE_REF_ERR_* flags.  The oracle
 * never allocates more than O(E) scratch and never aborts.
 *
 * Parity pins: every function here is pinned by tests that do not call it
 * to compute their expected values (brute force, closed forms, library
 * special cases, invariants); none is "parity unpinned".
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_REF_OK              0
#define MOE_REF_ERR_ARG         1   /* bad sizes or null pointers           */
#define MOE_REF_ERR_EXPERT_ID   2   /* an id outside [-1, E) was seen        */
#define MOE_REF_ERR_CAPACITY    4   /* more (t, r) pairs than capacity rows  */

/* fp32 -> bf16, round to nearest, ties to even (IEEE 754 binary32 -> bfloat16). */
uint16_t moe_ref_bf16_encode(float v);
float    moe_ref_bf16_decode(uint16_t b);

/* fp32 -> OCP FP8 E4M3 ("fn" variant), round to nearest even, saturating to
 * +-448; NaN -> 0x7F; the sign of zero is kept. */
uint8_t  moe_ref_e4m3_encode(float v);
float    moe_ref_e4m3_decode(uint8_t q);

/* Routing layout.  Inputs: topk_idx [T,K] (-1 = masked entry), topk_w [T,K]
 * (may be NULL: expert_weight is then left untouched).  Outputs (all caller
 * owned): tokens_per_expert[E], expert_offset[E+1], tokens_per_rank[R],
 * rank_offset[R+1], recv_expert_offset[E+1], recv_slot[T,R] (-1 = token not
 * sent to that rank), expert_slot[T,K] (-1 = masked), recv_src_token
 * [capacity] (-1 past the last used row), expert_src_row[T*K] and
 * expert_weight[T*K] (-1 / 0 past the last valid entry).  Ids outside
 * [-1, E) are flagged and treated as masked. */
int moe_ref_layout(const int32_t* topk_idx, const float* topk_w,
                   int32_t T, int32_t K, int32_t E, int32_t R, int64_t capacity,
                   int32_t* tokens_per_expert, int32_t* expert_offset,
                   int32_t* tokens_per_rank, int32_t* rank_offset,
                   int32_t* recv_expert_offset, int32_t* recv_slot,
                   int32_t* expert_slot, int32_t* recv_src_token,
                   int32_t* expert_src_row, float* expert_weight);

/* Multi-source receive layout: the single-GPU stand-in for the exchange in
 * which every source rank sends its tokens to the ranks of their experts and
 * every destination rank receives from all sources ("Inside the Nebius +
 * PyTorch DeepSeek V3 recipe", section "Mixture-of-experts and wide expert
 * parallelism").  S sources hold Ts tokens each; token g of the concatenated
 * routing topk_idx [T,K], T = S*Ts, belongs to source g / Ts.  Destination r
 * owns the receive region [r*T, (r+1)*T) (its worst case: every token of
 * every source); the tokens reaching r fill it from its start in (source,
 * token) order, which is ascending g.  Outputs:
 *   recv_slot[g,r]            r*T + #{g' < g : g' has a valid expert on r}, or -1
 *   tokens_per_rank[r]        rows used in region r
 *   rank_offset[R+1]          r*T (region starts); rank_offset[R] = R*T
 *   recv_source_offset[R,S+1] #{g < s*Ts : g reaches r}: source s's rows in
 *                             region r are [offset[r,s], offset[r,s+1]) from
 *                             the region start; offset[r,S] = tokens_per_rank[r]
 *   recv_src_token[R*T]       g of each used row, -1 in every region's tail
 * and the expert-major outputs exactly as moe_ref_layout defines them over
 * the T tokens (expert_src_row maps through this recv_slot). */
int moe_ref_layout_sources(const int32_t* topk_idx, const float* topk_w,
                           int32_t S, int32_t Ts, int32_t K, int32_t E, int32_t R,
                           int32_t* tokens_per_expert, int32_t* expert_offset,
                           int32_t* tokens_per_rank, int32_t* rank_offset,
                           int32_t* recv_source_offset, int32_t* recv_slot,
                           int32_t* expert_slot, int32_t* recv_src_token,
                           int32_t* expert_src_row, float* expert_weight);

/* bf16 dispatch: recv_x[recv_slot[t,r], :] = x[t, :] for every recv_slot >= 0.
 * x [T,H] and recv_x [capacity,H] hold bf16 bit patterns. */
int moe_ref_dispatch_bf16(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                          const int32_t* recv_slot, int64_t capacity,
                          uint16_t* recv_x);

/* FP8 dispatch: per token and 128-column block, scale and E4M3 codes as
 * described above, written to every destination row.  H % 128 == 0.
 * recv_q [capacity,H] bytes, recv_scales [capacity,H/128] fp32. */
int moe_ref_dispatch_fp8(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                         const int32_t* recv_slot, int64_t capacity,
                         uint8_t* recv_q, float* recv_scales);

/* MXFP8 dispatch (OCP Microscaling, E4M3 elements, E8M0 shared scale):
 * per token and 1x32 block, shared_exp = floor(log2(amax)) - 8 (8 is the
 * exponent of E4M3's largest normal, 448 = 1.75 * 2^8), clamped to
 * [-127, 127]; an all-zero block takes -127.  Scale byte = shared_exp + 127;
 * q = E4M3_RNE_satfinite(x * 2^-shared_exp).  H % 32 == 0.
 * recv_q [capacity,H] bytes, recv_scales [capacity,H/32] bytes. */
int moe_ref_dispatch_mxfp8(const uint16_t* x, int32_t T, int32_t H, int32_t R,
                           const int32_t* recv_slot, int64_t capacity,
                           uint8_t* recv_q, uint8_t* recv_scales);

/* Combine: out[t,:] = bf16_rne( fp32 fma chain over k ascending of
 * topk_w[t,k] * y[expert_slot[t,k], :] ), skipping expert_slot < 0.
 * y [n_rows,H] bf16 bits (expert-major), out [T,H] bf16 bits. */
int moe_ref_combine(const uint16_t* y, int64_t n_rows, int32_t T, int32_t K,
                    int32_t H, const int32_t* expert_slot, const float* topk_w,
                    uint16_t* out);

/* Low-latency dispatch (DeepEP's low-latency family, "Inside the Nebius +
 * PyTorch DeepSeek V3 recipe", section "DeepEP"): every valid entry (t,k) is
 * written to a fixed-capacity per-expert buffer recv [E, cap, H] at row
 * e * cap + j, j = #{(t',k') < (t,k) : idx[t',k'] == e}; entries with
 * j >= cap are dropped (ll_slot -1, MOE_REF_ERR_CAPACITY).  Outputs:
 * tokens_per_expert[E] (rows written), ll_slot[T,K] (row or -1).  Rows of
 * recv that receive nothing keep their contents.  The combine for this layout
 * is moe_ref_combine with ll_slot as the slot map. */
int moe_ref_ll_dispatch(const uint16_t* x, const int32_t* topk_idx, int32_t T, int32_t K, int32_t E,
                        int32_t H, int32_t cap, uint16_t* recv, int32_t* tokens_per_expert,
                        int32_t* ll_slot);

/* Backward of the bf16 dispatch (its adjoint): grad_x[t,:] = bf16_rne(fp32
 * sum over r ascending of grad_recv[recv_slot[t,r], :]), skipping slots < 0;
 * 0 for a token sent nowhere.  grad_recv [n_rows,H], grad_x [T,H] bf16 bits. */
int moe_ref_dispatch_backward(const uint16_t* grad_recv, int64_t n_rows, int32_t T, int32_t R,
                              int32_t H, const int32_t* recv_slot, uint16_t* grad_x);

/* Backward of combine: grad_y[expert_slot[t,k], :] = bf16_rne(fp32(topk_w[t,k]
 * * grad_out[t,:])) and grad_w[t,k] = sum_h grad_out[t,h] * y[expert_slot[t,k],h]
 * accumulated in double (masked entries: 0).  grad_out [T,H], y and grad_y
 * [n_rows,H] bf16 bits; grad_w [T,K] double. */
int moe_ref_combine_backward(const uint16_t* grad_out, const uint16_t* y, int64_t n_rows, int32_t T,
                             int32_t K, int32_t H, const int32_t* expert_slot, const float* topk_w,
                             uint16_t* grad_y, double* grad_w);

#ifdef __cplusplus
}
#endif
#endif /* MOE_ORACLE_H */
