/*
 * libspecverify: the speculative-sampling verify step on one GB300 (sm_103a).
 *
 * The operation (velog article "6-1편. Speculative Decoding", §2 "4-step algorithm" steps 3-4,
 * §2-1 accept/reject rule, §2-2 corrected distribution and sampling; greedy variant from
 * "All About Transformer Inference", Appendix D "Speculative Sampling", steps 1-3; the bonus token
 * from "Accelerating Sonar through speculation", §"Speculative decoding"):
 *
 *   for every sequence b of a CSR-packed batch, with gamma_b drafted tokens x_0..x_{gamma_b - 1}:
 *     p_i = softmax(target_logits[row t0 + i] / T)   for i = 0..gamma_b      (gamma_b + 1 rows)
 *     q_i = softmax(draft_logits[row d0 + i] / T)    for i = 0..gamma_b - 1  (gamma_b rows)
 *     accept x_i while u_i * q_i(x_i) < p_i(x_i)  (probability min(1, p/q)), in slot order;
 *     at the first rejected slot n draw a token from norm(max(0, p_n - q_n));
 *     if all gamma_b drafts are accepted (n = gamma_b) draw a bonus token from p_gamma.
 *   Draws use the inverse CDF in vocabulary index order: the smallest k whose running weight sum
 *   exceeds u' * (total weight); if rounding leaves none, the last k with positive weight.
 *   Greedy (T == 0): accept x_i while it equals argmax(target row t0 + i) (lowest index on ties);
 *   emit that argmax at the first mismatch, or argmax(target row t0 + gamma_b) when all match.
 *   Uniforms: u = (Philox4x32-10(ctr, key).word0 >> 8) * 2^-24 with key = (seed lo32, seed hi32) and
 *   ctr = (step lo32, step hi32, b, (slot << 8) | purpose), purpose 0 for the accept test of slot
 *   i and 1 for the draw at the emitting slot; b is the global sequence index.
 *
 * Layout (all row-major, row stride V elements, no padding):
 *   seq_offsets  int32[B + 1], seq_offsets[0] = 0, seq_offsets[b+1] - seq_offsets[b] = gammas[b].
 *   draft rows of b: seq_offsets[b] .. seq_offsets[b+1] - 1           (R_d = seq_offsets[B] rows)
 *   target rows of b: seq_offsets[b] + b .. seq_offsets[b+1] + b        (R_t = R_d + B rows)
 *   draft_tokens int32[R_d], aligned with the draft rows.
 *   out_tokens   int32[R_t], aligned with the target rows: slot j of b at seq_offsets[b] + b + j holds
 *                x_j for j < n, the drawn token at j = n, and -1 for n < j <= gamma_b.
 *   out_num_accepted int32[B]: n for every sequence, -1 for a sequence that failed a device check.
 *
 * Ownership and errors: every array argument is a DEVICE pointer owned by the caller; the library
 * never frees or retains them. Host-side argument errors return SV_ERR_INVALID_ARG (or
 * SV_ERR_WORKSPACE) before anything is launched. Data errors found on the device set bit
 * (1u << code) of the device status word. Inconsistent CSR offsets (seq_offsets[0] != 0, a gap
 * that differs from gammas[b], a negative gamma or one above max_gamma) fail the whole batch before
 * any logit row is read: every out_num_accepted is -1 and out_tokens is not written. A draft token
 * outside [0, V), a NaN or +inf logit, or a row whose logits are all -inf (-inf entries are
 * otherwise allowed and mean p = 0) fail only their sequence: its out_num_accepted is -1 and its
 * out_tokens slots are -1. No device check traps. Every wait of one warp on another within the launch
 * is bounded: a wait that gives up sets SV_ERR_TIMEOUT and fails the sequence it waited for in the
 * same way (n = -1, tokens -1; with the fused update its history and length are left unchanged and
 * its next token is -1). A sampled sequence's outputs have one writer, chosen by an atomic claim, so
 * a failed sequence's outputs are never overwritten by a late writer.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1, /* bad scalar, NULL pointer, misaligned pointer, unsupported size */
    SV_ERR_CUDA = 2,        /* a CUDA runtime call or launch failed */
    SV_ERR_BAD_TOKEN = 3,   /* device: draft token outside [0, V) */
    SV_ERR_BAD_OFFSETS = 4, /* device: seq_offsets / gammas inconsistent or gamma > max_gamma */
    SV_ERR_NONFINITE = 5,   /* device: NaN or +inf logit in a row the step reads */
    SV_ERR_EMPTY_ROW = 6,   /* device: a row whose logits are all -inf */
    SV_ERR_TIMEOUT = 7,     /* device: a bounded wait between warps of the launch gave up */
    SV_ERR_WORKSPACE = 8,   /* workspace NULL or smaller than spec_verify_workspace_size() */
    SV_ERR_CAPACITY = 9     /* device (spec_verify_commit): a sequence's history would overflow */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

/* Largest gamma_b one call accepts: the accept decisions of a sequence are one warp's lanes. */
#define SV_MAX_GAMMA 31

/*
 * Optional intermediate values (every field a nullable DEVICE pointer). Rows are numbered target
 * rows first (0 .. R_t - 1) then draft rows (R_t .. R_t + R_d - 1).
 *   row_lse    double[R_t + R_d]: log sum_k exp(l_k / T) of each row (sampling mode only).
 *   row_argmax int32[R_t]: argmax of each target row, lowest index on ties (greedy mode only).
 *   p_x, q_x   double[R_d]: p_i(x_i) and q_i(x_i) of every draft slot (sampling mode only).
 *   seq_mass   double[B]: total weight S of the sequence's draw relative to p (1 - beta at a
 *              rejected slot; about 1 for a bonus draw) (sampling mode only).
 *   beta       double[R_d]: beta_i = sum_x min(p_i(x), q_i(x)) of every draft slot, the acceptance
 *              probability of slot i when x_i is drawn from q_i (velog "6-1편. Speculative Decoding",
 *              §2-3); p_i(x_i) for a point-mass draft (sampling mode only). Computed by a second kernel
 *              enqueued after the step, from the logits.
 *   spin_limit polls after which a wait of one warp on another warp's word gives up (SV_ERR_TIMEOUT);
 *              0 keeps the library's bound (about a second). A small value exists to exercise the
 *              time-out path in tests: a sequence whose wait gave up reports n = -1 and tokens -1.
 *   order      the order of the statistics stream, for tests of both paths (the outputs are the same):
 *              0 the library's choice; 1 sequence order; 2 slot order wherever the call allows it (bf16
 *              rows on 16-byte boundaries, sampling with draft rows, linear drafts, none of the per-row
 *              fields above, B < 1024 and B (2 max_gamma + 1) <= 2048), whatever the batch's size.
 *   cluster    the small-batch form, for tests (the outputs are the same): 0 the library's choice (sampled
 *              batches small enough that the persistent launch would give each streaming warp at most one
 *              statistics task run one CTA cluster of up to 8 CTAs per sequence; greedy batches keep the
 *              persistent launch); 1 never; 2 wherever the call allows it, greedy included (linear drafts,
 *              none of the array fields above, V <= 131072, B clusters fit the SMs).
 */
typedef struct {
    double* row_lse;
    int32_t* row_argmax;
    double* p_x;
    double* q_x;
    double* seq_mass;
    double* beta;
    uint32_t spin_limit;
    uint32_t order;
    uint32_t cluster;
} sv_debug;

/*
 * The plain form: bf16 logits, the legacy default stream, blocking. It allocates its own
 * workspace and device status word, waits for the step to finish and returns SV_OK or the first
 * device error code (priority BAD_OFFSETS, BAD_TOKEN, NONFINITE, EMPTY_ROW, TIMEOUT, CAPACITY). Host sizes
 * are read from gammas (copied to the host once) to size the workspace. temperature == 0 selects
 * greedy, in which case draft_logits may be NULL and is never read.
 */
int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V,
                float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
                int32_t* out_num_accepted);

/* Bytes of device workspace spec_verify_ex needs for B sequences of gamma_b <= max_gamma over a
 * vocabulary of V. Returns 0 for invalid sizes. */
size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t max_gamma);

/*
 * The full form: asynchronous on `cuda_stream` (a cudaStream_t; NULL = legacy default stream), no
 * allocation and no host synchronisation. Requirements checked on the host: B >= 0, V >= 1,
 * 0 <= max_gamma <= SV_MAX_GAMMA, temperature finite and >= 0 with log2(e) / temperature finite in
 * float32 when positive, non-NULL target_logits / seq_offsets / gammas / draft_tokens / outputs,
 * non-NULL draft_logits when temperature > 0, workspace of at least
 * spec_verify_workspace_size(B, V, max_gamma) bytes aligned to 256 bytes. Rows may be at any
 * element alignment; 16-byte-aligned rows take the vectorised path. device_status (nullable) is a
 * device uint32 that the call ORs error bits into; the caller clears it. The workspace must not be
 * shared by calls that may overlap on the GPU. Returns SV_OK once the work is enqueued.
 */
int spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                   const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                   int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed,
                   uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                   uint32_t* device_status, void* workspace, size_t workspace_bytes,
                   const sv_debug* debug, void* cuda_stream);

/*
 * One contiguous range of a larger batch (a batch split over GPUs by sequence, or over calls): exactly
 * spec_verify_ex, with seq_base the index in the whole batch of this call's sequence 0. The uniforms of
 * sequence b are keyed by seq_base + b (mod 2^32), so verifying the ranges [s0, s1) of a batch, each with
 * seq_base = s0, and concatenating their outputs gives the whole batch's outputs (the draws of a sequence
 * depend only on its own rows and its global index). spec_verify_ex is this call with seq_base = 0.
 */
int spec_verify_range(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                      int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed,
                      uint64_t step, uint32_t seq_base, int32_t* out_tokens, int32_t* out_num_accepted,
                      uint32_t* device_status, void* workspace, size_t workspace_bytes,
                      const sv_debug* debug, void* cuda_stream);

/*
 * Device staging buffers of spec_verify_host, sized by the caller for the batch: target_logits
 * R_t x V elements, draft_logits R_d x V (may be NULL when the host call passes no draft logits),
 * draft_tokens R_d, seq_offsets B + 1, gammas B, out_tokens R_t, out_num_accepted B (R_d =
 * seq_offsets[B], R_t = R_d + B). Alignment rules as for spec_verify_ex's device arguments.
 */
typedef struct {
    void* target_logits;
    void* draft_logits;
    int32_t* draft_tokens;
    int32_t* seq_offsets;
    int32_t* gammas;
    int32_t* out_tokens;
    int32_t* out_num_accepted;
} sv_device_buffers;

/*
 * Host-buffer form: the step on inputs and outputs in host memory ("Accelerating Sonar through
 * speculation", §"Speculative decoding": the target model's logits for the gamma + 1 positions are
 * verified and the accepted tokens returned to the caller). On `cuda_stream`, in this order: the inputs
 * are copied from host memory into the staging buffers `dev`, the step runs as spec_verify_ex on them,
 * and the tokens and accepted counts are copied back to out_tokens / out_num_accepted in host memory.
 * With page-locked host memory every copy is asynchronous and the outputs are valid once the stream has
 * synchronised; with pageable memory the CUDA runtime may synchronise inside the copies. seq_offsets[B]
 * is read on the host to size the copies (SV_ERR_INVALID_ARG unless 0 <= seq_offsets[B] <=
 * B * max_gamma); the device still checks the whole CSR structure. Every argument check of
 * spec_verify_ex runs on the staging buffers before anything is enqueued. The host arrays, staging
 * buffers and workspace must stay valid until the stream has passed the call's work. The library owns
 * none of the buffers.
 */
int spec_verify_host(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                     const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas, int32_t B,
                     int32_t V, int32_t max_gamma, float temperature, uint64_t seed, uint64_t step,
                     int32_t* out_tokens, int32_t* out_num_accepted, const sv_device_buffers* dev,
                     uint32_t* device_status, void* workspace, size_t workspace_bytes, void* cuda_stream);

/*
 * Allocation-free form, for callers that cannot call cudaMalloc (for example code running inside a
 * stream capture it does not own, or a runtime without a device allocator). The pages describe no
 * such entry point; it exists for those callers only. It behaves as spec_verify_ex on the same
 * arguments, but its scratch is a fixed 8 MiB array compiled into the library (held on every GPU that
 * loads the library until the process exits) instead of a caller workspace. It allocates and frees
 * nothing. Batches whose spec_verify_workspace_size(B, V, max_gamma) exceeds 8 MiB are rejected with
 * SV_ERR_WORKSPACE before anything is launched. The first call on a device looks up the array's
 * device address (cudaGetSymbolAddress with that device current) and keeps it for that device; make
 * that first call before any stream capture. The kept address belongs to the device's primary
 * context as it was at that first call: after cudaDeviceReset, or from a different (non-primary)
 * context on the same device, it is no longer valid, and this entry point must not be used there. All calls share the one array and each call clears what it needs at its start, so
 * calls that may overlap on the GPU (other streams, other threads) race and must be serialised by the
 * caller.
 */
int spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                        const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                        int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed,
                        uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                        uint32_t* device_status, const sv_debug* debug, void* cuda_stream);

/*
 * Post-verify update on the device ("Accelerating Sonar through speculation", §"MTP scheduling": once
 * the drafts are verified, a kernel shifts the target's input tokens and inserts the next target token,
 * so the host does not have to wait for the accepted length before the next step is issued). Enqueued
 * on `cuda_stream` after spec_verify_ex on the same stream, it consumes that call's outputs on the
 * device; nothing is copied to the host and the host does not synchronise.
 *
 *   for every sequence b with n = out_num_accepted[b] >= 0 and L = lengths[b]:
 *     history[b * capacity + L + j] = out_tokens[seq_offsets[b] + b + j]   for j = 0..n
 *     lengths[b] = L + n + 1;  next_tokens[b] = out_tokens[seq_offsets[b] + b + n]
 *   (the n accepted drafts and the drawn token are appended; the drawn token is the next step's input
 *   token, at position lengths[b] - 1).
 *   A sequence with n < 0 (it failed verification) is left unchanged and gets next_tokens[b] = -1.
 *   A sequence with n > seq_offsets[b+1] - seq_offsets[b] or n > SV_MAX_GAMMA (outputs no verify call
 *   writes) or with L < 0 or
 *   L + n + 1 > capacity is left unchanged, gets next_tokens[b] = -1, and sets bit
 *   (1u << SV_ERR_BAD_OFFSETS) or (1u << SV_ERR_CAPACITY) of *device_status (if not NULL).
 *
 * Arguments: out_tokens int32[seq_offsets[B] + B], out_num_accepted int32[B] and seq_offsets
 * int32[B + 1] as spec_verify_ex wrote / read them; history int32[B * capacity], one row of capacity
 * tokens per sequence; lengths int32[B] (read and updated); next_tokens int32[B] (written). All are
 * DEVICE pointers owned by the caller, 4-byte aligned. Returns SV_ERR_INVALID_ARG for B < 0,
 * capacity < 1 or a NULL / misaligned pointer (B > 0), SV_ERR_CUDA if the launch fails, else SV_OK
 * (asynchronously: device-side findings go to *device_status).
 */
int spec_verify_commit(const int32_t* out_tokens, const int32_t* out_num_accepted, const int32_t* seq_offsets,
                       int32_t B, int32_t* history, int32_t capacity, int32_t* lengths, int32_t* next_tokens,
                       uint32_t* device_status, void* cuda_stream);

/*
 * The verify step with the post-verify update fused into it: spec_verify_ex on the same arguments
 * (without debug output) followed by the update spec_verify_commit describes, done inside the verify
 * launch by the warp that writes each sequence's final token, so no second kernel is launched. History,
 * lengths and next tokens follow spec_verify_commit; a sequence that fails verification keeps its
 * history and length and gets next token -1. Returns SV_ERR_INVALID_ARG for capacity < 1 or a NULL /
 * misaligned history, lengths or next_tokens (B > 0), else as spec_verify_ex.
 */
int spec_verify_fused(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                      int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed, uint64_t step,
                      int32_t* out_tokens, int32_t* out_num_accepted, uint32_t* device_status, void* workspace,
                      size_t workspace_bytes, int32_t* history, int32_t capacity, int32_t* lengths,
                      int32_t* next_tokens, void* cuda_stream);

/*
 * N-gram drafter (velog "6-1편. Speculative Decoding", §"drafter types", N-gram: no draft model; the
 * tokens that followed an earlier occurrence of the most recent n tokens are reused as the guess). For
 * every sequence b, with L = lengths[b] tokens history[b * capacity + 0 .. L-1]:
 *   for n = n_max down to n_min (the first n that matches): the largest s with s + n < L and
 *   history[s .. s+n-1] == history[L-n .. L-1]; the draft is the tokens history[s+n .. s+n+gamma-1],
 *   gamma = min(gamma_max, L - (s + n)), and match_pos[b] = s + n. No match: gamma 0, match_pos = L.
 * Outputs, CSR-packed as spec_verify_ex reads them: gammas[b], seq_offsets[0..B] (prefix sums of the
 * gammas) and draft_tokens[seq_offsets[b] .. seq_offsets[b+1]-1]. Such drafts have no draft
 * distribution: verify them with draft_logits NULL (point-mass drafts).
 * Arguments: history int32[B * capacity] and lengths int32[B] as spec_verify_commit maintains them
 * (1 <= capacity <= 32768); 1 <= n_min <= n_max; 0 <= gamma_max <= SV_MAX_GAMMA; draft_tokens
 * int32[B * gamma_max]; gammas and match_pos int32[B]; seq_offsets int32[B + 1]. All DEVICE pointers
 * owned by the caller, 4-byte aligned. A length outside [0, capacity] gives that sequence no draft and
 * sets (1u << SV_ERR_INVALID_ARG) in *device_status (if not NULL). Two launches on cuda_stream; returns
 * SV_ERR_INVALID_ARG for bad scalars or pointers, SV_ERR_CUDA if a launch fails, else SV_OK.
 */
int spec_draft_ngram(const int32_t* history, int32_t capacity, const int32_t* lengths, int32_t B, int32_t n_min,
                     int32_t n_max, int32_t gamma_max, int32_t* draft_tokens, int32_t* gammas,
                     int32_t* seq_offsets, int32_t* match_pos, uint32_t* device_status, void* cuda_stream);

/*
 * Token-tree verification with point-mass candidates. The pages sketch tree drafts (EAGLE's top-K
 * candidates: "Accelerating Sonar through speculation", §"EAGLE") but give no rule; the reading here
 * applies velog "6-1편. Speculative Decoding" §2-1/§2-2 to the children of the current node, each a point
 * mass:
 *   cur = root; at node cur its children are tried in index order; child c with token x is accepted iff
 *   u_c * (1 - P_E) < p_cur(x), where P_E is the p_cur mass of the distinct tokens rejected before it
 *   (a repeated token is rejected); the first accepted child's token is emitted and the walk moves to
 *   it; if no child is accepted (or cur is a leaf), the last token is drawn from p_cur with the rejected
 *   tokens removed (if that leaves no mass, from p_cur), and the walk stops. The emitted tokens are then
 *   distributed exactly as sampling from the target. Greedy (T == 0): the first child whose token is the
 *   argmax of the current row is taken; else that argmax is emitted.
 * Layout: the CSR of spec_verify_ex with gamma_b = the number of non-root nodes of tree b (<= 31):
 *   node 0 is the root, node j >= 1 is draft slot seq_offsets[b] + j - 1 with token draft_tokens[.] and
 *   parent parents[.] in [0, j); target row seq_offsets[b] + b + j holds the logits after the path to
 *   node j. Uniforms: the accept test of node j uses slot j - 1 (purpose 0), the final draw at node cur
 *   uses slot cur (purpose 1): a chain (parents of slot i = i) verifies exactly as spec_verify_ex with
 *   point-mass drafts (draft_logits NULL).
 * Outputs: out_tokens[seq_offsets[b] + b + j] for j <= n: the accepted path's tokens, then the drawn
 * one (-1 after); out_num_accepted[b] = n; out_path (nullable, int32[R_d]) [seq_offsets[b] + j] = the
 * j-th accepted node for j < n, -1 after. A parent outside [0, j) fails its sequence
 * (SV_ERR_BAD_OFFSETS); other errors as spec_verify_ex. Workspace: spec_verify_workspace_size.
 */
int spec_verify_tree(const void* target_logits, sv_dtype dtype, const int32_t* draft_tokens, const int32_t* parents,
                     const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                     float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                     int32_t* out_path, uint32_t* device_status, void* workspace, size_t workspace_bytes,
                     void* cuda_stream);

/*
 * Vocabulary-sharded verify ("All About Transformer Inference", the model-parallel sections: the logits
 * come out of an unembedding sharded over the vocabulary across tensor-parallel ranks; "Accelerating Sonar
 * through speculation", the tensor-parallel scheduling section). Shard j of S holds columns
 * [bounds[j], bounds[j+1]) of every target and draft row as its own row-major arrays of
 * Vs = bounds[j+1] - bounds[j] columns (bounds[0] = 0, bounds[S] = V, S <= 8). The step is the
 * unsharded one (same rule, same uniforms, same outputs up to the rounding order of the sums), run as
 * four calls per shard with three exchanges between the shards (all-gathers over the tensor-parallel
 * group; a caller running the shards in one process concatenates the records instead):
 *   1. spec_shard_stats   per row, the statistics of the shard's slice      -> sv_shard_partial[rows]
 *      exchange 1: all-gather the partials into [S][rows] (rows = R_t + R_d, targets first; R_t alone
 *      in greedy mode or with point-mass drafts)
 *   2. spec_shard_decide  the merged statistics, the accept tests and the first rejection (every shard
 *      computes the same): writes out_num_accepted, the accepted tokens and -1 past the emitting slot
 *      (greedy: the whole output), and each sequence's draw           -> sv_shard_draw[B]
 *   3. spec_shard_sums    per sequence and SV_SHARD_CHUNK-column chunk of the slice, the draw's exact
 *      sums (4 float pairs)                                           -> float[B][NC][4][2]
 *      exchange 2: all-gather the sums into [S][B][NC][4][2]; NC = spec_shard_chunks(S, bounds), the
 *      chunk count of the widest shard (a narrower shard's records past its slice are zero)
 *   4. spec_shard_finish  the (shard, chunk) holding the draw's target u S, found from the gathered sums;
 *      that shard scans the chunk and writes the drawn token (a global column) at the emitting slot,
 *      every other shard writes -1 there
 *      exchange 3: element-wise max of out_tokens over the shards (the drawn slot); every other entry is
 *      the same on all shards.
 * All arrays are DEVICE pointers owned by the caller: partial, draw and sums arrays 16-byte aligned, the rest
 * 4-byte aligned. draft_tokens, seq_offsets and gammas are the unsharded batch's, identical on every
 * shard; shard_draft is NULL in greedy mode or for point-mass drafts (then point_mass = 1 at T > 0).
 * Data errors go to *device_status as in spec_verify_ex (pass the same word to stats and decide; a bad
 * CSR structure fails every sequence). Each call is asynchronous on cuda_stream; returns
 * SV_ERR_INVALID_ARG for bad scalars or pointers, SV_ERR_CUDA if a launch fails, else SV_OK.
 */
#define SV_SHARD_CHUNK 8192 /* columns per sums record */

typedef struct {
    float m;     /* raw maximum of the slice's logits (NaN: a NaN or +inf logit in the slice) */
    float s;     /* sum over the slice of 2^((l - m) log2(e) / T) (sampling) */
    int32_t arg; /* first argmax of the slice as a global column, -1 if none */
    float g;     /* the logit at the row's draft token if this shard holds that column, else 0 */
} sv_shard_partial;

typedef struct {
    int32_t words[8]; /* one sequence's draw (mode, emitting slot, row maxima, ratio, uniform), opaque */
} sv_shard_draw;

int spec_shard_stats(const void* shard_target, const void* shard_draft, sv_dtype dtype, const int32_t* draft_tokens,
                     const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t v0, int32_t Vs,
                     int32_t max_gamma, float temperature, void* partials, uint32_t* device_status, void* cuda_stream);

/* shard_bounds_host: a HOST array of S + 1 columns (see above). */
int spec_shard_decide(const void* all_partials, int32_t S, const int32_t* shard_bounds_host, const int32_t* draft_tokens,
                      const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                      float temperature, int32_t point_mass, uint64_t seed, uint64_t step, int32_t* out_tokens,
                      int32_t* out_num_accepted, void* draws, uint32_t* device_status, void* cuda_stream);

/* Records per sequence and shard in the sums: ceil(max_j (bounds[j+1] - bounds[j]) / SV_SHARD_CHUNK), or 0
 * for bounds that are not S + 1 increasing columns from 0 with S <= 8 (a host call). */
int32_t spec_shard_chunks(int32_t S, const int32_t* shard_bounds_host);

int spec_shard_sums(int32_t shard, int32_t S, const int32_t* shard_bounds_host, const void* shard_target,
                    const void* shard_draft, sv_dtype dtype, const void* draws, const int32_t* seq_offsets, int32_t B,
                    int32_t V, float temperature, void* sums, void* cuda_stream);

int spec_shard_finish(int32_t shard, int32_t S, const int32_t* shard_bounds_host, const void* shard_target,
                      const void* shard_draft, sv_dtype dtype, const void* draws, const void* all_sums,
                      const int32_t* seq_offsets, int32_t B, int32_t V, float temperature, int32_t* out_tokens,
                      void* cuda_stream);

/* Map a device status word (OR of 1u << code) to one status code, by the priority above. */
int spec_verify_status_from_bits(uint32_t bits);

/* Static, human-readable name of a status code. */
const char* spec_verify_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
