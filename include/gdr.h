/*
 * gdr.h -- C ABI of libgdr, the gated delta rule forward on GB300 (sm_103a).
 *
 * The operation (Kev-4B-LiteRT page "r15_kernel_test.py", function truth_f64; DEG page
 * "model.py", function delta_rule_reference): per row and value head h, with key head
 * hk = h / (Hv/Hk) (adjacent value heads share a key head, repeat_interleave order),
 *
 *   k^ = k / sqrt(sum k^2 + 1e-6),  q~ = q / sqrt(sum q^2 + 1e-6) * D^-0.5
 *   S = S0 (zeros if absent); for each token t:
 *     S = exp(g_t) S;  delta = beta_t (v_t - S^T k^);  S = S + k^ delta^T;  o_t = S^T q~
 *
 * Pads are data: a position with beta = g = 0 neither decays nor writes the state.
 *
 * Conventions shared by every call:
 *  - All array pointers are DEVICE pointers owned by the caller, row-major and contiguous,
 *    16-byte aligned. The library never allocates device memory; scratch memory, where a path
 *    needs it, is a caller-provided workspace.
 *  - D = Dk = Dv must be 128 (GDR_ERR_UNSUPPORTED otherwise). Hv must be a multiple of Hk.
 *  - q, k, v and o share one element type (gdr_dtype); g, beta and every state are float32.
 *  - Calls are asynchronous on `stream` (NULL = the legacy default stream). Host-side argument
 *    checks happen before anything is launched and return an error without touching the GPU.
 *    Errors found on the device (a fork index out of range, a wait that ran out) are recorded
 *    in a sticky device error word that gdr_sync_status() reads and clears.
 *  - No exception crosses the ABI; every call returns a gdr_status. gdr_last_error_message()
 *    gives a one-line reason for the last non-OK status returned on the calling host thread.
 */
#ifndef GDR_H
#define GDR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GDR_OK = 0,
  GDR_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment, workspace too small  */
  GDR_ERR_UNSUPPORTED = 2,   /* a size the kernels do not implement (D != 128)            */
  GDR_ERR_CUDA = 3,          /* a CUDA runtime call failed (launch, sync, encode)          */
  GDR_ERR_DEVICE_INDEX = 4,  /* a fork's trunk index was outside [0, N)                    */
  GDR_ERR_TIMEOUT = 5        /* a kernel wait ran past its limit; the kernel stopped early */
} gdr_status;

typedef enum { GDR_F32 = 0, GDR_BF16 = 1 } gdr_dtype;

/* Same type as cudaStream_t, declared here so that C callers need no CUDA header. */
typedef struct CUstream_st* gdr_stream_t;

/*
 * Workspace bytes gdr_chunk_fwd needs for these sizes (0 when the path needs none: float32, and
 * rows of one chunk, L <= 64, which the bfloat16 path finishes in a single kernel). For longer
 * rows the bfloat16 tensor-core path keeps per-chunk intermediates there (the factors M', N, Q',
 * P U of each 64-token chunk). Returns 0 for invalid sizes.
 */
size_t gdr_chunk_workspace_bytes(int B, int L, int Hk, int Hv, int D, gdr_dtype dt);

/*
 * Prefill: B rows of L tokens each, every row continuing its own initial state.
 * (Kev-4B-LiteRT "r15_kernel_test.py": kernel(q, k, v, g, beta, initial_state,
 *  output_final_state=True, use_qk_l2norm_in_kernel=True) -> (o, S_T);
 *  DEG "model.py", _delta_rule.)
 *   q, k   [B, L, Hk, D]  dt          raw (not yet normalised) queries and keys
 *   v      [B, L, Hv, D]  dt
 *   g      [B, L, Hv]     float32     natural-log decay per token and value head (<= 0)
 *   beta   [B, L, Hv]     float32     write strength
 *   S0     [B, Hv, D, D]  float32     initial state, S[i][j] = key i, value j; NULL = zeros
 *   o      [B, L, Hv, D]  dt          output, every position (pads included)
 *   S_T    [B, Hv, D, D]  float32     final state; NULL = not written. May alias S0.
 *   ws     workspace of at least gdr_chunk_workspace_bytes(...) bytes (may be NULL if that is 0)
 * L need not be a multiple of 64; nothing is written beyond position L-1.
 */
gdr_status gdr_chunk_fwd(const void* q, const void* k, const void* v, const float* g,
                         const float* beta, const float* S0, void* o, float* S_T, int B, int L,
                         int Hk, int Hv, int D, gdr_dtype dt, void* ws, size_t ws_bytes,
                         gdr_stream_t stream);

/*
 * Prefill of B right-padded rows of different lengths (DEG "model.py": Backbone.forward over a batch
 * whose State.lengths give each row's real tokens; _dn_gates makes the padding exact no-ops).
 * Same arguments, layouts, workspace and results as gdr_chunk_fwd, plus
 *   lengths [B] int32 (device)   valid tokens of each row, in [0, L]
 * Row b runs only its first lengths[b] tokens: positions at or past lengths[b] are pads whatever
 * their g and beta hold, the 64-token chunks wholly past it are skipped (no work), o is not written
 * there (it keeps what the caller left), and S_T[b] is the state after the row's last valid token
 * (S0[b] when the length is 0). A length outside [0, L] leaves that row's o and S_T untouched and
 * records GDR_ERR_DEVICE_INDEX in the device error word.
 */
gdr_status gdr_chunk_fwd_varlen(const void* q, const void* k, const void* v, const float* g,
                                const float* beta, const float* S0, const int32_t* lengths, void* o,
                                float* S_T, int B, int L, int Hk, int Hv, int D, gdr_dtype dt, void* ws,
                                size_t ws_bytes, gdr_stream_t stream);

/*
 * Prefill followed by the layer's gated RMSNorm, fused into the output of the recurrence (DEG
 * "model.py": _linear_layer applies _gated_rms with the in_proj_z gate to _delta_rule's output). Same
 * arguments, workspace and final state as gdr_chunk_fwd, but instead of o it writes
 *   out[b, t, h, :] = w * o / sqrt(mean(o^2) + eps) * silu(z[b, t, h, :]),  silu(x) = x / (1 + exp(-x))
 * over the 128 values of each position and value head, from the float32 o (o itself is not stored):
 *   z    [B, L, Hv, D] bfloat16   the gate; 16-byte aligned
 *   w    [D] float32              the norm weight; 16-byte aligned
 *   eps  >= 0
 *   out  [B, L, Hv, D] bfloat16   must not overlap z
 * bfloat16 only (GDR_ERR_UNSUPPORTED for float32). Rows of several chunks reduce over the four
 * column blocks of a head in the state kernel (a cluster of four CTAs); rows of one chunk (L <= 64)
 * run gdr_gated_rmsnorm over the bf16 o in place.
 */
gdr_status gdr_chunk_fwd_gated(const void* q, const void* k, const void* v, const float* g,
                               const float* beta, const float* S0, const void* z, const float* w, float eps,
                               void* out, float* S_T, int B, int L, int Hk, int Hv, int D, gdr_dtype dt, void* ws,
                               size_t ws_bytes, gdr_stream_t stream);

/* Bytes of caller workspace gdr_fork_fwd needs for these sizes (0 for float32, and 0 for
 * single-chunk forks, L_pad <= 64, which the tensor-core path finishes in one kernel). */
size_t gdr_fork_workspace_bytes(int F, int L_pad, int Hk, int Hv, int D, gdr_dtype dt);

/*
 * Fork batch: F forks, fork f continuing its own copy of trunk[trunk_idx[f]] over its L_pad
 * tokens (right-padded with beta = g = 0). The trunk states are read in place, never copied.
 * bf16 forks run on the same tensor-core kernels as gdr_chunk_fwd (one row per fork, the row's
 * initial state taken from the trunk by index), so fork f equals gdr_chunk_fwd on that row from
 * trunk[trunk_idx[f]] bit for bit; float32 forks run the token loop.
 * (DEG "model.py": fork_delta_rule(q, k, v, g, beta, h0, h0_idx, store) in _fork_linear_layer;
 *  Backbone.fork reads the prefixes by reference through the row index prow.)
 *   q, k        [F, L_pad, Hk, D] dt;  v [F, L_pad, Hv, D] dt;  g, beta [F, L_pad, Hv] float32
 *   trunk       [N, Hv, D, D] float32   shared prefix states
 *   trunk_idx   [F] int64 (device)      fork f starts from trunk[trunk_idx[f]]
 *   o           [F, L_pad, Hv, D] dt
 *   states_out  [F, Hv, D, D] float32   each fork's final state (the `store` of the pages);
 *                                       NULL = not kept. Must not overlap trunk.
 *   ws          workspace of at least gdr_fork_workspace_bytes(...) bytes (NULL if that is 0),
 *               owned by the caller and free for reuse once the call's stream work is done
 * An index outside [0, N) leaves that fork's outputs untouched and records
 * GDR_ERR_DEVICE_INDEX in the device error word.
 */
gdr_status gdr_fork_fwd(const void* q, const void* k, const void* v, const float* g,
                        const float* beta, const float* trunk, const int64_t* trunk_idx, int N,
                        void* o, float* states_out, int F, int L_pad, int Hk, int Hv, int D,
                        gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream);

/*
 * One decode step (L = 1) for F rows, each row's state updated in place.
 * (DEG "model.py": DecodeGraph.step -> fork_forward(keep=True, decode=True); an idle row has
 *  lens 0, hence beta = g = 0, and its state stays bit-identical.)
 *   q, k [F, 1, Hk, D] dt;  v [F, 1, Hv, D] dt;  g, beta [F, 1, Hv] float32
 *   states [F, Hv, D, D] float32, read and written in place;  o [F, 1, Hv, D] dt
 */
gdr_status gdr_decode_step(const void* q, const void* k, const void* v, const float* g,
                           const float* beta, float* states, void* o, int F, int Hk, int Hv,
                           int D, gdr_dtype dt, gdr_stream_t stream);

/*
 * Prefill without a caller workspace and without any device allocation. The pages have no
 * counterpart to this call; it is for callers that cannot allocate GPU memory: a host program
 * that owns the whole device memory budget (a serving process or engine that reserves the GPU at
 * start-up, or a plugin loaded into one), or a latency-critical loop where a cudaMalloc, which may
 * synchronise the device and can fail under memory pressure, is not allowed once running.
 *
 * Same arguments (minus ws and ws_bytes), computation, results and errors as gdr_chunk_fwd. The
 * scratch is a fixed array of GDR_NOALLOC_SCRATCH_BYTES in device memory, held by every GPU on which
 * the library's code is loaded until the process exits. Sizes whose workspace
 * (gdr_chunk_workspace_bytes) exceeds it are rejected with GDR_ERR_UNSUPPORTED and a message, before
 * any CUDA call; float32 q/k/v need no scratch.
 * The first call on a device looks up the scratch's device address (with that device current);
 * make that first call before any stream capture. The address belongs to the device's CUDA
 * context: after that context is destroyed (cudaDeviceReset) the next call looks it up again in
 * the new one, so that call too belongs before any capture.
 * Every call uses the same scratch, which keeps the previous call's contents (nothing in it needs
 * to start at zero: each call writes all the scratch it reads). Calls whose GPU work overlaps
 * (other streams, other host threads) race on the scratch: serialise them.
 */
#define GDR_NOALLOC_SCRATCH_BYTES ((size_t)64 * 1024 * 1024)
gdr_status gdr_chunk_fwd_noalloc(const void* q, const void* k, const void* v, const float* g,
                                 const float* beta, const float* S0, void* o, float* S_T, int B,
                                 int L, int Hk, int Hv, int D, gdr_dtype dt, gdr_stream_t stream);

/*
 * GDN prologue: from the layer's q|k|v projection to the path's inputs.
 * (DEG "model.py": _linear_layer with _conv_silu and _dn_gates.) Per row b, with
 * ext = [tail; mixed] along positions (K-1 carried inputs, then the L new ones) and
 * C = (2 Hk + Hv) D channels,
 *   y[t][c] = silu( sum_{j < K} conv_w[c][j] ext[t + j][c] ),  silu(x) = x / (1 + exp(-x))
 * split by channel into q (channels [0, Hk D)), k ([Hk D, 2 Hk D)) and v (the rest), and
 *   beta = sigmoid(b),  g = -exp(A_log[h]) softplus(a + dt_bias[h])   at valid positions t < len_b,
 *   beta = g = 0 at pads (positions >= len_b), so that pads are exact no-ops of the recurrence;
 *   new_tail[b][j] = ext[len_b + j] for j < K-1 (the inputs ending at the last valid token).
 * q, k and v are computed at every position, pads included (their values there do not matter).
 *   mixed    [B, L, C] bfloat16           the projection
 *   tail     [B, K-1, C] bfloat16         the previous call's carry; NULL = zeros (a new sequence)
 *   conv_w   [C, K] float32               depthwise causal weights; tap K-1 meets the current token
 *                                         (16-byte aligned, like mixed, tail, q, k, v and new_tail)
 *   a, b     [B, L, Hv] float32           decay and write-strength projections
 *   A_log, dt_bias [Hv] float32
 *   lengths  [B] int32 (device)           valid tokens per row, in [0, L]; NULL = L for every row.
 *                                         A length outside [0, L] leaves that row's g, beta and
 *                                         new_tail untouched and records GDR_ERR_DEVICE_INDEX.
 *   q, k     [B, L, Hk, D] bfloat16;  v [B, L, Hv, D] bfloat16
 *   g, beta  [B, L, Hv] float32
 *   new_tail [B, K-1, C] bfloat16         NULL = not written; must not overlap tail or mixed
 * K is the convolution width, 1 <= K <= 8 (the pages use 4); B <= 65535 and L <= 1048560
 * (GDR_ERR_UNSUPPORTED otherwise). Arithmetic is float32 from the
 * bfloat16 inputs, with one rounding of q, k, v to bfloat16.
 */
gdr_status gdr_prologue(const void* mixed, const void* tail, const float* conv_w, const float* a,
                        const float* b, const float* A_log, const float* dt_bias, const int32_t* lengths,
                        void* q, void* k, void* v, float* g, float* beta, void* new_tail, int B, int L,
                        int Hk, int Hv, int D, int K, gdr_stream_t stream);

/*
 * The GDN prologue fused into the bfloat16 prefill: gdr_prologue (K = 4, lengths NULL) followed by
 * gdr_chunk_fwd on its q, k, v, g and beta, without q, k, v, g and beta ever reaching memory
 * (DEG "model.py": _linear_layer, where _conv_silu and _dn_gates feed _delta_rule). The chunk
 * kernel forms each 64-token tile of q, k and v as the conv + SiLU of the projection rows (and the
 * carry) in gdr_prologue's own order of operations, one rounding to bfloat16, and each chunk's g and
 * beta from a and b the same way: for rows longer than one chunk (L > 64) o, S_T and new_tail equal
 * those of the two separate calls bit for bit; rows of one chunk take the two-kernel path (which
 * gdr_chunk_fwd replaces by one kernel), equal within the bf16 tolerance, new_tail bit for bit.
 *   mixed, tail, conv_w, a, b, A_log, dt_bias, new_tail   as for gdr_prologue (conv_w [C, 4]; tail
 *                                   NULL = zeros, new_tail NULL = not written)
 *   S0, o, S_T                      as for gdr_chunk_fwd with dt = GDR_BF16 (o [B, L, Hv, D] bf16)
 *   ws    workspace of at least gdr_chunk_fwd_prologue_workspace_bytes(...) bytes (never NULL,
 *         every L included), owned by the caller: the per-chunk factors
 * o and new_tail must overlap neither mixed, tail nor each other. K must be 4 and D 128
 * (GDR_ERR_UNSUPPORTED otherwise); B, Hv <= 65535. Every row has L valid tokens (for rows with their
 * own lengths, call gdr_prologue with lengths and then gdr_chunk_fwd_varlen).
 */
size_t gdr_chunk_fwd_prologue_workspace_bytes(int B, int L, int Hk, int Hv, int D, int K);
gdr_status gdr_chunk_fwd_prologue(const void* mixed, const void* tail, const float* conv_w, const float* a,
                                  const float* b, const float* A_log, const float* dt_bias, const float* S0,
                                  void* o, float* S_T, void* new_tail, int B, int L, int Hk, int Hv, int D,
                                  int K, void* ws, size_t ws_bytes, gdr_stream_t stream);

/*
 * Gated RMSNorm epilogue: per row of D values (a position and value head of the recurrence
 * output o [B, L, Hv, D], so rows = B L Hv), with the gate z of the same shape,
 *   out = w * (x / sqrt(mean(x^2) + eps)) * silu(z),   silu(z) = z / (1 + exp(-z))
 * (DEG "model.py": _gated_rms, applied to the output of _delta_rule with the in_proj_z gate.)
 *   x, z, out  [rows, D] bfloat16   out may be x or z itself, but may not partly overlap them
 *   w          [D] float32          the norm weight (16-byte aligned, like x, z and out)
 * D must be 128; eps >= 0; rows <= 2^34. Arithmetic is float32 from the bfloat16 inputs, one
 * rounding of out.
 */
gdr_status gdr_gated_rmsnorm(const void* x, const void* z, const float* w, float eps, void* out,
                             long long rows, int D, gdr_stream_t stream);

/*
 * Backward of gdr_chunk_fwd: the gradients of a loss with respect to every input, given its
 * gradients dO of the outputs o and dS_T of the final state. The pages train through the
 * recurrence (DEG "model.py", delta_rule_reference inside the training loss; Kev-4B-LiteRT
 * "r15_kernel_test.py", truth_f64) but print no backward; this is the plain reverse of the
 * forward stated at the top of this header, token by token:
 *   dq~ = S_t dO_t;  dS += q~ dO_t^T;  dk^ = dS delta;  ddelta = dS^T k^;  dbeta = ddelta . (v - kv);
 *   dv = beta ddelta;  dkv = -beta ddelta;  dS_a = dS + k^ dkv^T;  dk^ += S_a dkv;
 *   dg = <S_a, dS_a>;  dS = exp(g_t) dS_a
 * (S_a = exp(g_t) S_{t-1}, kv = S_a^T k^), from dS = dS_T at the last token; dS0 is the last dS;
 * dq and dk are taken back through the normalisations and summed over the value heads of a key
 * head. Pads are tokens like any other (their dv is 0 because beta = 0).
 *   q, k, v, g, beta, S0     as for gdr_chunk_fwd (S0 NULL = zeros)
 *   dO     [B, L, Hv, D]  dt        gradient of o
 *   dS_T   [B, Hv, D, D]  float32   gradient of the final state; NULL = zeros
 *   dq, dk [B, L, Hk, D]  float32;  dv [B, L, Hv, D] float32;  dg, dbeta [B, L, Hv] float32
 *   dS0    [B, Hv, D, D]  float32   gradient of S0; NULL = not written
 *   ws     workspace of at least gdr_backward_workspace_bytes(...) bytes (never NULL), owned by
 *          the caller: state checkpoints every 32 tokens, one 32-token segment of states per
 *          (row, value head, 16-column block), and the per-column-block partial sums
 * The outputs must not overlap the inputs or one another. Arithmetic is float32 throughout (the
 * states are recomputed from checkpoints by the forward's own float32 recurrence), and the sums
 * over column blocks and value heads run in a fixed order: the result is deterministic.
 * B <= 65535 and B L < 2^31 (GDR_ERR_UNSUPPORTED otherwise).
 */
size_t gdr_backward_workspace_bytes(int B, int L, int Hk, int Hv, int D);
gdr_status gdr_backward(const void* q, const void* k, const void* v, const float* g, const float* beta,
                        const float* S0, const void* dO, const float* dS_T, float* dq, float* dk,
                        float* dv, float* dg, float* dbeta, float* dS0, int B, int L, int Hk, int Hv,
                        int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream);

/*
 * gdr_backward_chunked: the same gradients as gdr_backward for bf16 q, k, v, dO, computed chunk by
 * chunk on the tensor cores. The pages print no backward; this is the reverse of the chunked
 * forward (the chunk algebra of gdr_chunk_fwd, 64-token chunks): the sequential part is the
 * adjoint chain, the forward chain transposed,
 *   dS_c = Gamma_C dS_{c+1} + M'^T dS_{c+1} + Q'^T dO_c    (dS_NC = dS_T, dS0 = dS_0),
 * and the rest is local to each chunk once its entering state S_c and dS_{c+1} are known (the
 * gradients through Delta = U - W S, P, T = (I + A)^-1, the decays and the normalisations).
 * Arguments, shapes, ownership and the no-overlap rule as for gdr_backward; dt must be GDR_BF16
 * (GDR_ERR_UNSUPPORTED otherwise). ws holds at least gdr_backward_chunked_workspace_bytes(...)
 * bytes: the forward's per-chunk factors and the chunk-entry states and adjoints (fp16 with a power
 * of two per 32-column slice, 32 KiB per row, value head and chunk each). The products
 * take fp16 (bf16 for the raw q, k Gram products) operands with float32 accumulation, like the
 * bf16 forward, so the result matches the float64 backward to the bf16 path's tolerance, not
 * gdr_backward's float32 one; the sums run in a fixed order (deterministic).
 */
size_t gdr_backward_chunked_workspace_bytes(int B, int L, int Hk, int Hv, int D);
gdr_status gdr_backward_chunked(const void* q, const void* k, const void* v, const float* g, const float* beta,
                                const float* S0, const void* dO, const float* dS_T, float* dq, float* dk,
                                float* dv, float* dg, float* dbeta, float* dS0, int B, int L, int Hk, int Hv,
                                int D, gdr_dtype dt, void* ws, size_t ws_bytes, gdr_stream_t stream);

/*
 * The chunked backward without its recomputation, for callers that keep the forward's
 * intermediates instead of checkpointing (the DEG model recomputes them; both give the same
 * gradients). gdr_chunk_fwd_save is gdr_chunk_fwd for bf16 rows (o and S_T as gdr_chunk_fwd
 * computes them for rows longer than one chunk, bit for bit; rows of one chunk take the two-kernel
 * path, equal within the bf16 tolerance) that also leaves in `saved` what gdr_backward_chunked's
 * sequential forward passes would recompute: the per-chunk factors, the fp16 chunk-entry states
 * with their powers of two, and v's powers of two. gdr_backward_chunked_saved then runs only the
 * adjoint chain and the chunk-local gradients; its results equal gdr_backward_chunked's bit for bit.
 *   saved  at least gdr_backward_chunked_workspace_bytes(B, L, Hk, Hv, D) bytes, 16-byte aligned,
 *          owned by the caller, overlapping no input or output. Between the two calls it must stay
 *          untouched and the backward must be given the same q, k, v, g, beta and S0 (nothing
 *          checks this: other inputs give wrong gradients, not an error).
 * Arguments, sizes and checks otherwise as gdr_chunk_fwd (dt = GDR_BF16) and gdr_backward_chunked.
 */
gdr_status gdr_chunk_fwd_save(const void* q, const void* k, const void* v, const float* g, const float* beta,
                              const float* S0, void* o, float* S_T, int B, int L, int Hk, int Hv, int D,
                              gdr_dtype dt, void* saved, size_t saved_bytes, gdr_stream_t stream);
gdr_status gdr_backward_chunked_saved(const void* q, const void* k, const void* v, const float* g,
                                      const float* beta, const float* S0, const void* dO, const float* dS_T,
                                      float* dq, float* dk, float* dv, float* dg, float* dbeta, float* dS0, int B,
                                      int L, int Hk, int Hv, int D, gdr_dtype dt, void* saved, size_t saved_bytes,
                                      gdr_stream_t stream);

/* Synchronise `stream`, then read and clear the sticky device error word of the current device. */
gdr_status gdr_sync_status(gdr_stream_t stream);

/*
 * Testing aid (failure detection): the SM clock cycles a kernel wait may take before the kernel
 * gives up, records GDR_ERR_TIMEOUT in the device error word, waits (again bounded) for its own
 * copies and products still in flight, frees its tensor memory and exits. Default about 2e9
 * cycles (roughly 1 s); 0 makes every wait that is not already satisfied give up at once; a
 * negative value restores the default. Applies to launches made after the call; results of a call
 * that timed out are undefined, and the next call runs normally.
 */
gdr_status gdr_debug_set_wait_budget(long long cycles);

/* Static strings; never NULL. */
const char* gdr_status_string(gdr_status status);
const char* gdr_last_error_message(void);

/*
 * Stage timer (measurement aid). When enabled, every kernel the library launches is bracketed
 * by a pair of CUDA events recorded on its launch stream (up to `capacity` launches).
 * gdr_stage_timer_collect() synchronises those events and, for each kernel id k < max_ids,
 * writes the summed milliseconds to total_ms[k] and the launch count to launches[k], then
 * clears the record. gdr_kernel_name(k) names kernel id k (NULL past the last id).
 */
gdr_status gdr_stage_timer_enable(int on, int capacity);
gdr_status gdr_stage_timer_collect(double* total_ms, int* launches, int max_ids);
const char* gdr_kernel_name(int id);

#ifdef __cplusplus
}
#endif

#endif /* GDR_H */
