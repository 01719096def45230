/*
 * rm_cp.h -- C ABI of the GB300 (sm_103a) chunkwise gated linear attention
 * library, organised around per-segment affine state summaries.
 *
 * Method, per batch row b and head h (q_t, k_t in R^Dk, v_t in R^Dv, g_t a
 * scalar gate, alpha_t = exp(g_t), or 0 when token t starts a sequence):
 *     S_t = alpha_t S_{t-1} + k_t v_t^T,      o_t = scale * S_t^T q_t.
 * The sequence axis is cut into num_segments equal contiguous segments, the
 * "shards" of the Megatron-Core API docs page
 * "core.ssm.context_parallel.chunkwise"; here all of them live on one GPU and
 * no collective is involved.  The six compute calls follow that page's
 * LinearAttentionCPBackend protocol and its two drivers:
 *
 *   forward   rm_cp_forward_prepare  -> (M, delta_S) per segment   [cp_forward_prepare]
 *             rm_cp_compose_prefix   -> S_in per segment            [chunkwise_cp_forward]
 *             rm_cp_forward_apply    -> o                           [cp_forward_apply]
 *   backward  rm_cp_backward_prepare -> gamma per segment (+ dq)    [cp_backward_prepare]
 *             rm_cp_compose_suffix   -> dS_out per segment          [chunkwise_cp_backward]
 *             rm_cp_backward_apply   -> dk, dv, dg                  [cp_backward_apply]
 *
 * Conventions for every call:
 *   - Layouts are contiguous row-major: q, k, dq, dk [B,T,H,Dk]; v, o, dO, dv
 *     [B,T,H,Dv]; g, dg [B,T,H] (fp32); summaries [nseg,B,H,Dk,Dv] (fp32);
 *     M [nseg,B,H] (fp32).  With vector gates (rm_cp_problem.vector_gates)
 *     g, dg are [B,T,H,Dk] and M is [nseg,B,H,Dk].  Segment j covers tokens
 *     [j*L, (j+1)*L) of every row, L = T / num_segments.
 *   - q, k, v, o, dO, dq, dk, dv have the problem's dtype (RM_F32 or RM_BF16;
 *     bf16 results are rounded to nearest even from fp32).  g, dg, M and all
 *     summaries are always fp32.
 *   - Every pointer passed to a compute call is a DEVICE pointer, 16-byte
 *     aligned, owned by the caller.  The library never allocates, frees or
 *     synchronises; it only enqueues kernels on the given stream (0 = the
 *     legacy default stream).  Outputs are fully overwritten.
 *   - All validation happens on the host before anything is launched.  On a
 *     non-OK status nothing was enqueued; rm_cp_last_error() returns a
 *     thread-local description.  Launch failures map to RM_ERR_CUDA, and the
 *     description names the CUDA error of the launch that failed.  A compute
 *     call first makes the current device's primary context current on the
 *     calling thread (a thread that has made no CUDA call yet may have none)
 *     and clears a non-sticky CUDA error that an earlier runtime call left
 *     pending on that thread (cudaGetLastError is per thread), so that only
 *     its own launches decide its status.  Kernels contain no traps and no
 *     inter-block waits.
 *   - Calls are thread-safe; concurrent calls on different streams may not
 *     share output buffers.
 */
#ifndef RM_CP_H
#define RM_CP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without requiring cuda_runtime.h */
typedef struct CUstream_st* rm_stream_t;

typedef enum {
    RM_OK = 0,
    RM_ERR_INVALID_ARG = 1, /* null pointer, non-positive size, bad enum          */
    RM_ERR_SHAPE = 2,       /* T % num_segments, (T/nseg) % chunk, size overflow  */
    RM_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned                   */
    RM_ERR_UNSUPPORTED = 4, /* head dims outside the supported set                */
    RM_ERR_METADATA = 5,    /* cu_seqlens not 0 = cu[0] < ... < cu[n] = T          */
    RM_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed               */
    RM_ERR_TIMEOUT = 7      /* reserved for bounded device-side waits             */
} rm_status;

typedef enum { RM_F32 = 0, RM_BF16 = 1 } rm_dtype;

/*
 * Problem description shared by all calls.
 *   B, T, H, Dk, Dv  batch rows, tokens per row, heads, key and value dims.
 *                    Supported: Dk in {16, 32, 64, 128}; Dv a multiple of 8
 *                    in [8, 256].
 *   num_segments     contiguous segments per row; T % num_segments == 0.
 *   chunk            the chunk length of the chunkwise form; the segment
 *                    length must be a multiple of it.  The result does not
 *                    depend on it beyond rounding: kernels block the
 *                    sequence axis in tiles of their own.
 *   scale            output scale (commonly 1/sqrt(Dk)); passed explicitly.
 *   seq_idx          NULL: every row is one sequence.  Otherwise a device
 *                    int32 [T] array of non-decreasing sequence ids
 *                    (PackedSequenceCPMetadata.local_seq_idx, concatenated
 *                    over segments), applied to every row; token t starts a
 *                    sequence when t == 0 or seq_idx[t] != seq_idx[t-1].
 *   preceding_start  NULL (all prefixes start at segment 0) or device int32
 *                    [num_segments]: inclusive first segment of segment j's
 *                    forward-summary prefix (preceding_rank_start).
 *   following_stop   NULL (all suffixes end at num_segments) or device int32
 *                    [num_segments]: exclusive end of segment j's
 *                    backward-summary suffix (following_rank_stop).
 *   q_heads          0 (or H): q holds one row per head, [B,T,H,Dk].  Else
 *                    a divisor of H: q is [B,T,q_heads,Dk] and head h reads
 *                    q row h / (H / q_heads), i.e. consecutive heads share
 *                    their queries (as the heads of a Mamba2 group share C).
 *                    dq stays [B,T,H,Dk]: one gradient per head.
 *   vector_gates     0: one gate per (token, head) as above.  1: one gate per
 *                    (token, head, key dimension): g, dg are [B,T,H,Dk]
 *                    fp32 and S_t = diag(alpha_t) S_{t-1} + k_t v_t^T with
 *                    alpha_t[i] = exp(g_t[i]) (all 0 at a sequence start).
 *                    The segment transition is then the diagonal matrix
 *                    M = diag(prod of alpha) -- the general M of the page's
 *                    CPForwardUnpackedSummary (S_out = M S_in + delta_S),
 *                    M^T = M -- stored as its diagonal, M [nseg,B,H,Dk]; the
 *                    compositions apply it row by row, and the workspace
 *                    holds one fp32 value per (row, token, head, key
 *                    dimension).  bf16 storage with Dk = Dv = 128 runs on
 *                    the tensor cores; other shapes and fp32 storage on the
 *                    generic fp32-arithmetic kernels.
 * Out-of-range metadata values are clamped on the device to [0, j] and
 * [j+1, num_segments]; rm_cp_build_packed_metadata produces valid ones.
 */
typedef struct {
    int32_t B, T, H, Dk, Dv;
    int32_t num_segments;
    int32_t chunk;
    float scale;
    rm_dtype dtype;
    const int32_t* seq_idx;
    const int32_t* preceding_start;
    const int32_t* following_stop;
    int32_t q_heads;
    int32_t vector_gates;
} rm_cp_problem;

/*
 * Host helper: rank-local packed-sequence metadata for every segment
 * (PackedSequenceCPMetadata / build_packed_sequence_cp_metadata on the
 * Megatron-Core page).  All arrays are HOST memory owned by the caller.
 *   cu_seqlens_host       [num_seqs+1], 0 = cu[0] < cu[1] < ... < cu[num_seqs] = T
 *   seq_idx_host          out [T]: i for cu[i] <= t < cu[i+1]
 *   local_cu_seqlens_host out, concatenated per segment: 0, every sequence
 *                         start strictly inside the segment (relative to the
 *                         segment start), then L.  Capacity needed:
 *                         num_seqs + 2*num_segments entries.
 *   local_cu_offsets_host out [num_segments+1]: segment j's entries are
 *                         [off[j], off[j+1]).
 *   preceding_start_host  out [num_segments]: segment holding the start of
 *                         the sequence that holds segment j's first token.
 *   following_stop_host   out [num_segments]: 1 + segment holding the last
 *                         token of the sequence that holds segment j's last
 *                         token.
 * Errors: RM_ERR_INVALID_ARG (null pointer, non-positive sizes),
 * RM_ERR_SHAPE (T % num_segments), RM_ERR_METADATA (bad cu_seqlens).
 */
rm_status rm_cp_build_packed_metadata(const int32_t* cu_seqlens_host, int32_t num_seqs,
                                      int32_t T, int32_t num_segments,
                                      int32_t* seq_idx_host,
                                      int32_t* local_cu_seqlens_host,
                                      int32_t* local_cu_offsets_host,
                                      int32_t* preceding_start_host,
                                      int32_t* following_stop_host);

/* Validate a problem without launching anything (RM_OK if every call accepts it). */
rm_status rm_cp_validate(const rm_cp_problem* p);

/*
 * Bytes of device workspace the calls need for this problem (0 if none; 0
 * also for an invalid problem).  The SAME workspace must be passed, unchanged
 * in between, to rm_cp_backward_prepare and the rm_cp_backward_apply that
 * follows it: the first leaves per-token partial gate gradients there for the
 * second.  rm_cp_forward_fused uses it during its own call only.  The
 * separate forward calls accept NULL.
 */
size_t rm_cp_workspace_size(const rm_cp_problem* p);

/*
 * cp_forward_prepare ("compute the local state summary with zero incoming
 * state"), for every segment at once.
 *   k [B,T,H,Dk], v [B,T,H,Dv] (dtype), g [B,T,H] fp32       in
 *   M [nseg,B,H] fp32: exp(sum of the segment's gates), or 0 when one of its
 *     tokens starts a sequence (its first token included)     out
 *   dS [nseg,B,H,Dk,Dv] fp32: the segment's end state from S_in = 0   out
 *   ws: unused (may be NULL).
 */
rm_status rm_cp_forward_prepare(const rm_cp_problem* p, const void* k, const void* v,
                                const float* g, float* M, float* dS, void* ws,
                                rm_stream_t stream);

/*
 * chunkwise_cp_forward's causal prefix: for every segment j,
 *   S_in[j] = sum_{i in [pre_j, j)} (M_{i+1} ... M_{j-1}) dS_i,
 * i.e. the summaries of segments pre_j .. j-1 (CPForwardUnpackedSummary:
 * S_out = M S_in + delta_S) applied in order to a zero state.
 *   M [nseg,B,H], dS [nseg,B,H,Dk,Dv] fp32 in;  S_in [nseg,B,H,Dk,Dv] fp32 out.
 */
rm_status rm_cp_compose_prefix(const rm_cp_problem* p, const float* M, const float* dS,
                               float* S_in, rm_stream_t stream);

/*
 * cp_forward_apply ("compose the preceding summaries and compute the local
 * output"): o_t for every token, each segment starting from its S_in.
 *   q, k [B,T,H,Dk], v [B,T,H,Dv] (dtype), g fp32, S_in fp32   in
 *   o [B,T,H,Dv] (dtype)                                        out
 *   ws: unused (may be NULL).
 */
rm_status rm_cp_forward_apply(const rm_cp_problem* p, const void* q, const void* k,
                              const void* v, const float* g, const float* S_in, void* o,
                              void* ws, rm_stream_t stream);

/*
 * The whole forward in one call: rm_cp_forward_prepare, rm_cp_compose_prefix
 * and rm_cp_forward_apply fused -- chunkwise_cp_forward's gather of the
 * preceding summaries done by each segment itself, cp_forward_apply's
 * "compose the preceding summaries and compute the local output".  Same
 * inputs and outputs as the three calls (M, dS, S_in and o are all written,
 * with the same values: the summaries are composed by the same chain of
 * multiply-adds), plus a workspace.
 *   On the tensor-core path (bf16, Dk = 128, Dv in {128, 256}) this is ONE
 *   kernel launch (plus a clear of the workspace's flags): every CTA
 *   prepares its segment's summary, then composes its own S_in from the
 *   summaries and inclusive prefixes other CTAs of the launch have published
 *   (a bounded look-back: CTAs start in segment order and wait, each wait
 *   bounded, only for segments that started earlier), then applies.  On the
 *   generic path it runs the three calls in order.
 *   ws: device workspace of rm_cp_workspace_size bytes (its content is
 *   overwritten; not needed across calls).
 *   Measured on GB300 this one launch is slower than the three calls on the
 *   configurations here: all CTAs of a wave finish their summaries together,
 *   so few find a predecessor's inclusive prefix already published, and each
 *   then folds the summaries of the segments before it (more bytes and more
 *   dependent loads than the separate, fully parallel composition).
 */
rm_status rm_cp_forward_fused(const rm_cp_problem* p, const void* q, const void* k,
                              const void* v, const float* g, float* M, float* dS, float* S_in,
                              void* o, void* ws, rm_stream_t stream);

/*
 * cp_backward_prepare ("compute local gamma with zero outgoing-state
 * gradient"), for every segment, for the loss L = sum_t dO_t . o_t:
 *   gamma_j = dL_j / dS_in[j] = sum over tokens t of segment j that belong to
 *             the sequence open at its first token a of
 *             (alpha_a ... alpha_t) * scale * q_t dO_t^T.
 * dq depends only on forward-direction states, all known once S_in is, so
 * this call also writes dq_t = scale * S_t dO_t and leaves q_t . dq_t per
 * token in the workspace for rm_cp_backward_apply.
 *   q, k [B,T,H,Dk], v, dO [B,T,H,Dv] (dtype), g fp32, S_in fp32   in
 *   gamma [nseg,B,H,Dk,Dv] fp32, dq [B,T,H,Dk] (dtype)             out
 *   ws: device workspace of rm_cp_workspace_size bytes             out
 */
rm_status rm_cp_backward_prepare(const rm_cp_problem* p, const void* q, const void* k,
                                 const void* v, const float* g, const float* S_in,
                                 const void* dO, float* gamma, void* dq, void* ws,
                                 rm_stream_t stream);

/*
 * chunkwise_cp_backward's reverse-causal suffix: for every segment j,
 *   dS_out[j] = sum_{i in (j, fol_j)} (M_{j+1} ... M_{i-1}) gamma_i,
 * i.e. CPBackwardUnpackedSummary dS_in = M^T dS_out + gamma (M is a scalar
 * per row and head here) applied from segment fol_j - 1 down to j + 1.
 *   M [nseg,B,H], gamma [nseg,B,H,Dk,Dv] fp32 in;  dS_out fp32 out.
 */
rm_status rm_cp_compose_suffix(const rm_cp_problem* p, const float* M, const float* gamma,
                               float* dS_out, rm_stream_t stream);

/*
 * cp_backward_apply ("compose the reverse-causal suffix and finish the local
 * input gradients"): dk, dv and dg of every token, each segment's adjoint
 * starting from dS_out[j] at its last token.
 *   dk_t = D_t v_t, dv_t = D_t^T k_t with D_t = scale q_t dO_t^T + alpha_{t+1} D_{t+1};
 *   dg_t = sum_{r >= t, same sequence} (q_r . dq_r - k_r . dk_r), exactly 0 at
 *          sequence starts; the part beyond the segment is <S_out, dS_out>,
 *          with S_out read as S_in[j+1] (equal to the segment's end state
 *          whenever dS_out[j] is not zero).
 *   q, k [B,T,H,Dk], v, dO [B,T,H,Dv] (dtype), g, S_in, dS_out fp32   in
 *   ws: the workspace rm_cp_backward_prepare filled                    in
 *   dk [B,T,H,Dk], dv [B,T,H,Dv] (dtype), dg [B,T,H] fp32             out
 */
rm_status rm_cp_backward_apply(const rm_cp_problem* p, const void* q, const void* k,
                               const void* v, const float* g, const void* dO,
                               const float* S_in, const float* dS_out, void* dk, void* dv,
                               float* dg, void* ws, rm_stream_t stream);

/*
 * Failure detection.  Every wait inside the tensor-core kernels (on a TMA
 * copy or on tensor-core completion) is bounded (200 ms); a wait that runs
 * out sets a device-side flag, and the kernel finishes its remaining work
 * with bounded waits and frees its tensor memory instead of hanging.
 *
 * rm_cp_device_status reads (and, if clear != 0, resets) that flag.  It
 * enqueues one tiny kernel and a copy on `stream`, then SYNCHRONISES the
 * stream (the only call of this library that does).  dev_scratch is a device
 * int32 the call may overwrite.  Returns RM_ERR_TIMEOUT if a wait ran out
 * since the flag was last cleared, RM_OK otherwise, RM_ERR_CUDA on a CUDA error.
 *
 * rm_cp_selftest_wait_timeout enqueues a one-thread kernel that waits on a
 * barrier nothing ever completes, with a bound of limit_us microseconds
 * (1 <= limit_us <= 1000000): it exercises the timeout path above without
 * faulting or hanging the device.  Returns RM_ERR_INVALID_ARG for an
 * out-of-range limit.
 */
rm_status rm_cp_device_status(int32_t* dev_scratch, int32_t clear, rm_stream_t stream);
rm_status rm_cp_selftest_wait_timeout(uint32_t limit_us, rm_stream_t stream);

/*
 * The whole backward in one call, with no device allocation and no
 * workspace argument: rm_cp_backward_prepare, rm_cp_compose_suffix and
 * rm_cp_backward_apply, in that order on `stream`, with the per-token
 * scratch they pass between each other taken from a fixed array that the
 * library itself holds in device memory.  The Megatron-Core page has no counterpart to
 * this call; it exists for callers that cannot allocate device memory, such
 * as a custom operator reached through a plugin interface with a fixed
 * signature and no workspace, or a deployment whose device memory is
 * planned up front and must not grow after start-up.
 *   Inputs, outputs and their layouts are those of the three calls it
 *   replaces: q, k, v, dO (dtype), g fp32, S_in and M from the forward;
 *   gamma and dS_out [nseg,B,H,Dk,Dv] fp32 are written as by those calls;
 *   dq, dk, dv (dtype), dg fp32 out.
 *   Limit: B * T * H <= 4,194,304 (16 MiB of fp32 scratch); larger
 *   problems get RM_ERR_SHAPE and must use the workspace form.
 *   The array is placed on a device when the library's code for this call
 *   is loaded there.  Under CUDA's default lazy module loading that happens
 *   in the first call on the device, which looks the array's device address
 *   up with that device current; the 16 MiB stay on the device until the
 *   process exits.  A caller whose memory plan is fixed at start-up should
 *   therefore make one call on each device during start-up, and before any
 *   stream capture (a module cannot be loaded during capture).  A failed
 *   lookup returns RM_ERR_CUDA, leaves no CUDA error pending, and is retried
 *   by the next call.  Every call shares the one array: calls whose work
 *   overlaps on the GPU (other streams, other host threads) race on it and
 *   must be serialised by the caller.  Nothing in the array needs clearing:
 *   each call writes every entry it later reads.
 */
rm_status rm_cp_backward_noalloc(const rm_cp_problem* p, const void* q, const void* k,
                                 const void* v, const float* g, const float* S_in,
                                 const float* M, const void* dO, float* gamma, float* dS_out,
                                 void* dq, void* dk, void* dv, float* dg, rm_stream_t stream);

/*
 * End to end from host memory: one step of the path (the three forward
 * calls, and the three backward calls when host->dO is not NULL) with its
 * inputs copied in from host buffers and its results copied back out, all
 * enqueued without blocking the host.  The Megatron-Core page has no counterpart to this
 * call; it is the step a training loop makes when its batches live in host
 * memory, with the copies of one step overlapping the kernels of the next.
 *
 *   Streams: the host-to-device copies go on h2d, the compute calls on
 *   compute, the device-to-host copies on d2h (one cudaMemcpyAsync per
 *   tensor).  Each device buffer set carries three events (cudaEvent_t,
 *   e.g. from rm_cp_event_create): `loaded` is recorded on h2d once the
 *   inputs are in, `computed` on compute after the last kernel, `drained` on
 *   d2h once the results are out.  Before reusing a set, h2d waits for the
 *   set's previous `computed` (its kernels have read the old inputs) and
 *   compute waits for its previous `drained` (its old results have left), so
 *   consecutive calls that alternate between two sets overlap the copies of
 *   one step with the kernels of another and never reuse a buffer early.
 *   An event never recorded counts as complete.
 *
 *   host: host buffers, laid out as on the device; page-locked (pinned) for
 *     the copies to run asynchronously.  q, k, v, g in; o out; for the
 *     backward dO in and dq, dk, dv, dg out (all NULL for a forward step).
 *   set:  device buffers of one step with the same fields, plus its events.
 *   st:   device buffers the compute calls pass between each other, shared by
 *     all sets (every compute call is on `compute`, so steps never overlap on
 *     them): M, dS, S_in, and for the backward gamma, dS_out and the
 *     workspace of rm_cp_workspace_size bytes.
 *   Everything is validated before anything is enqueued; a CUDA error on
 *   the copies or events returns RM_ERR_CUDA (work already enqueued stays).
 */
typedef struct {
    const void* q;
    const void* k;
    const void* v;
    const float* g;
    const void* dO;
    void* o;
    void* dq;
    void* dk;
    void* dv;
    float* dg;
} rm_cp_host_io;

typedef struct {
    void* q;
    void* k;
    void* v;
    float* g;
    void* dO;
    void* o;
    void* dq;
    void* dk;
    void* dv;
    float* dg;
    void* loaded;    /* cudaEvent_t */
    void* computed;  /* cudaEvent_t */
    void* drained;   /* cudaEvent_t */
} rm_cp_step_set;

typedef struct {
    float* M;
    float* dS;
    float* S_in;
    float* gamma;
    float* dS_out;
    void* ws;
} rm_cp_step_state;

rm_status rm_cp_step_host(const rm_cp_problem* p, const rm_cp_host_io* host,
                          const rm_cp_step_set* set, const rm_cp_step_state* st,
                          rm_stream_t compute, rm_stream_t h2d, rm_stream_t d2h);

/* A CUDA event without timing (cudaEventDisableTiming) on the current device,
 * for rm_cp_step_set; destroy it with rm_cp_event_destroy. */
rm_status rm_cp_event_create(void** event);
rm_status rm_cp_event_destroy(void* event);

/*
 * Mamba2 SSD scan on the same path.  The context-parallel pages name Mamba2
 * as the other user of exact state passing; its scan, per row b and head h,
 *     h_t = exp(dt_t A_h) h_{t-1} + dt_t B_t x_t^T,   y_t = h_t^T C_t + D_h x_t,
 * with B_t, C_t [N] shared by the H / G heads of a group (head h uses group
 * h / (H / G)), is the gated recurrence above with q = C, k = dt B, v = x,
 * g = dt A and scale 1.  These three calls map the SSD arguments onto the six
 * calls and map the results back; the problem passed to all of them has
 * Dk = N, Dv = P and scale = 1 (any other scale is RM_ERR_INVALID_ARG here).
 *   x, y, dy, dx [B,T,H,P] and Bm, Cm, dB, dC [B,T,G,N] have the problem's
 *   dtype; dt, ddt [B,T,H], A, D, dA, dD [H] are fp32.  G >= 1 divides H.
 *
 * rm_ssd_map_inputs: k [B,T,H,N] = dt B (rounded to the dtype), g [B,T,H] =
 *   dt A (fp32), and, when q is not NULL, q [B,T,H,N] = C of the head's group.
 *   v is x itself.  With q NULL (and Cm unused) the problem passed to the six
 *   calls sets q_heads = G and passes C itself as q: no copy of C per head.
 * rm_ssd_finish_forward: y = o + D_h x, in place over o (D may be NULL: o
 *   is then y already and nothing is enqueued).
 * rm_ssd_finish_backward: after the backward calls ran with dO = dy:
 *   dx = dv + D_h dy (in place over dv; D may be NULL), dC = sum over the
 *   group's heads of dq, dB = sum of dt dk, ddt = B . dk + A_h dg,
 *   dA_h = sum over (b, t) of dt dg, dD_h = sum of x . dy (the gradient at
 *   D = 0 when D is NULL).
 *   Sums run in a fixed order: the results do not depend on the launch.
 *   ws: device workspace of rm_ssd_workspace_size bytes.
 */
size_t rm_ssd_workspace_size(const rm_cp_problem* p);
rm_status rm_ssd_map_inputs(const rm_cp_problem* p, int32_t G, const float* dt, const float* A,
                            const void* Bm, const void* Cm, void* q, void* k, float* g,
                            rm_stream_t stream);
rm_status rm_ssd_finish_forward(const rm_cp_problem* p, const void* x, const float* D, void* o,
                                rm_stream_t stream);
rm_status rm_ssd_finish_backward(const rm_cp_problem* p, int32_t G, const void* x,
                                 const float* dt, const float* A, const void* Bm,
                                 const void* dy, const float* D, const void* dq, const void* dk,
                                 void* dv, const float* dg, float* ddt, float* dA, void* dB,
                                 void* dC, float* dD, void* ws, rm_stream_t stream);

/*
 * Gated delta rule on the same segment-summary path.  Per row b and head h,
 * with g_t and beta_t [B,T,H] fp32, alpha_t = exp(g_t) (0 when token t starts
 * a sequence) and A_t = alpha_t (I - beta_t k_t k_t^T):
 *     S_t = A_t S_{t-1} + beta_t k_t v_t^T,      o_t = scale S_t^T q_t.
 * A segment's summary is the Megatron-Core page's general affine map
 * S_out = M S_in + delta_S (CPForwardUnpackedSummary) with the Dk x Dk
 * transition M = A_last ... A_first (0 when a token of the segment starts a
 * sequence); the backward composes dS_in = M^T dS_out + gamma
 * (CPBackwardUnpackedSummary).  The six calls mirror the scalar-gate ones:
 *   rm_gdr_forward_prepare  M [nseg,B,H,Dk,Dk], dS [nseg,B,H,Dk,Dv] fp32 out
 *                           (and the per-chunk factors in ws, tensor cores)
 *   rm_gdr_compose_prefix   S_in[j] = fold over [pre_j, j) of S <- M_i S + dS_i
 *   rm_gdr_forward_apply    o
 *   rm_gdr_backward_prepare gamma [nseg,B,H,Dk,Dv] (the local adjoint at the
 *                           segment start, zero outgoing gradient) and
 *                           dq_t = scale S_t dO_t; saves states (every 16
 *                           tokens, every 64 on the tensor cores) in ws
 *   rm_gdr_compose_suffix   dS_out[j] = fold over (j, fol_j) of D <- M_i^T D + gamma_i
 *   rm_gdr_backward_apply   from D = dS_out at each segment's end:
 *                           dk, dv [B,T,H,*] (dtype), dg, dbeta [B,T,H] fp32
 *                           (dg exactly 0 at sequence starts)
 * The problem is an rm_cp_problem (vector_gates = 0, any q_heads): Dk in
 * {16, 32, 64, 128}, Dv a multiple of 8 up to 128, segment lengths a multiple of
 * 16 (RM_ERR_UNSUPPORTED otherwise).  bf16 storage with Dk = Dv = 64 and
 * segment lengths that are multiples of 64 runs the four sweeps on the
 * tensor cores in the chunkwise WY/UT form (per 64-token chunk the products
 * of the I - beta k k^T factors as one triangular solve); everything else,
 * and the two folds, on generic fp32-arithmetic kernels (at Dk = 128 a slow
 * fallback; with Dv > 64 there the backward apply runs its reverse sweep on
 * each half of the value columns in turn, and the workspace also holds the
 * first half's partial dk, dbeta and dg: B T H (Dk + 2) fp32 more).  ws:
 * rm_gdr_workspace_size bytes (B H (T / 16) Dk Dv fp32), one workspace for
 * the whole step, passed unchanged to every call that takes it: the backward
 * prepare saves states there for the backward apply (every 16 tokens, every
 * 64 on the tensor cores), and on the tensor cores the forward prepare also
 * leaves there each chunk's triangular factors T = (I + A)^-1 diag(beta) and
 * (I + A)^-1 (bf16; they depend on k, g and beta only), which the forward
 * apply and the two backward calls read, so the forward prepare must have run
 * on the same k, g, beta and ws before them (the generic kernels do not use
 * ws in the forward); the tensor-core backward apply also keeps each chunk's
 * state adjoint there between its two launches.  Validation, ownership and
 * errors as for the other calls.
 *
 * rm_gdr_path: 1 when the problem's sweeps run on the tensor cores, 0 on the
 * generic kernels, -1 for a problem these calls reject.
 */
int32_t rm_gdr_path(const rm_cp_problem* p);
size_t rm_gdr_workspace_size(const rm_cp_problem* p);
rm_status rm_gdr_forward_prepare(const rm_cp_problem* p, const void* k, const void* v,
                                 const float* g, const float* beta, float* M, float* dS, void* ws,
                                 rm_stream_t stream);
rm_status rm_gdr_compose_prefix(const rm_cp_problem* p, const float* M, const float* dS,
                                float* S_in, rm_stream_t stream);
rm_status rm_gdr_forward_apply(const rm_cp_problem* p, const void* q, const void* k, const void* v,
                               const float* g, const float* beta, const float* S_in, void* o, void* ws,
                               rm_stream_t stream);
rm_status rm_gdr_backward_prepare(const rm_cp_problem* p, const void* q, const void* k,
                                  const void* v, const float* g, const float* beta,
                                  const float* S_in, const void* dO, float* gamma, void* dq,
                                  void* ws, rm_stream_t stream);
rm_status rm_gdr_compose_suffix(const rm_cp_problem* p, const float* M, const float* gamma,
                                float* dS_out, rm_stream_t stream);
rm_status rm_gdr_backward_apply(const rm_cp_problem* p, const void* q, const void* k, const void* v,
                                const float* g, const float* beta, const void* dO,
                                const float* dS_out, void* dk, void* dv, float* dg, float* dbeta,
                                void* ws, rm_stream_t stream);

/* Name of a status code (static string). */
const char* rm_cp_status_string(rm_status s);

/* Thread-local detail for the last non-OK status returned on this thread. */
const char* rm_cp_last_error(void);

/* Number of kernels this library has enqueued in this process so far (all
 * devices, all threads).  A diagnostic for counting launches per step. */
uint64_t rm_cp_launch_count(void);

/* Which kernel family a problem runs on: 0 = generic SIMT fp32 path for
 * every call, 1 = tensor-core (tcgen05) path for every call, 2 = tensor-core
 * path for some calls and the generic path for the others.  -1 for an
 * invalid problem.  The tensor-core path serves bf16 storage with Dk = 128,
 * Dv in {128, 256} and segment lengths that are multiples of 64; with vector
 * gates, bf16 storage with Dk = Dv = 128 and segment lengths that are
 * multiples of 64 (other vector-gate problems run on the generic path). */
int32_t rm_cp_path(const rm_cp_problem* p);

#ifdef __cplusplus
}
#endif

#endif /* RM_CP_H */
