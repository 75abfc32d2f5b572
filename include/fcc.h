/*
 * fcc.h -- libfcc: GEMMs fused with the collective that consumes their output,
 * for one GB300 (sm_103a), across R tensor-parallel ranks whose buffers are
 * disjoint allocations in the one GPU's HBM.
 *
 * "Communication" between ranks is a kernel storing into (or loading from)
 * another rank's buffer.  The operators are the fused kernels named in
 * "GPU-vezerelt kommunikacioval gyorsitjak az AI-betanitast a kutatok"
 * (mKernel article, section on the five fused kernels: AllGather + GEMM,
 * GEMM + AllReduce, MoE Dispatch + GEMM, GEMM + ReduceScatter) and in
 * "Optimizing Distributed ML Communication with Fused Computation-Collective
 * Operations" (SC24, abstract: GEMV + AllReduce, GEMM + All-to-All, with
 * workgroups that ship their results as soon as they finish).
 *
 * Conventions for every call
 *  - Matrices are row-major and contiguous.  A_r is [M,K], B_r is [K,N]; the
 *    product is A_r @ B_r as in torch.  Shard j of an M-row result is the
 *    contiguous row block [j*M/R, (j+1)*M/R).
 *  - Pointer arrays (A, B, out, ...) are HOST arrays of DEVICE pointers, one
 *    per rank; they are read during the call and not retained.  Device
 *    pointers must be 16-byte aligned.  The caller owns every buffer.
 *  - Inputs are bf16; accumulation is f32; f32 results are stored as f32 and
 *    bf16 results are rounded to nearest even.
 *  - Calls are asynchronous on `stream` and return after enqueueing.
 *    Argument errors are reported synchronously and nothing is launched.
 *    Errors found on the device (a wait that timed out, a receive buffer too
 *    small) are recorded in a per-device status word that fcc_stream_status()
 *    reads and clears.
 *  - opts may be NULL for the defaults (fused, deterministic, library-owned
 *    workspace, 1 s wait limit).
 *  - Workspace: calls that need scratch memory take it from opts->workspace
 *    (size from fcc_workspace_size / fcc_moe_workspace_size); with no
 *    workspace given, the library keeps an internal per-device pool that it
 *    grows with cudaMalloc on first use (and when a larger call comes), which
 *    synchronises the device at that moment.
 *  - Not thread-safe for concurrent calls on the same stream; calls on
 *    different streams share the internal pool and must not overlap unless
 *    each passes its own workspace.
 *  - Environment defaults, read once when the library first needs one:
 *    FCC_ALGO=fused|unfused|interdecom|ce replaces FCC_ALGO_AUTO (also in
 *    fcc_choose_algo) for the operators with several forms (a form an
 *    operator lacks gives FCC_ERR_UNSUPPORTED; the attention and the MoE
 *    combine have one form and ignore it); FCC_DETERMINISTIC=0|1 is the
 *    summation mode of calls with opts == NULL; FCC_CHUNKS=n (1..64) the
 *    InterDecom chunk count where opts->chunks is 0; FCC_TIMEOUT_MS=n the
 *    device wait limit where opts->timeout_ns is 0.  Unset or unparsable
 *    values leave the built-in defaults.
 */
#ifndef FCC_H_
#define FCC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without pulling in the CUDA headers. */
typedef struct CUstream_st *fcc_stream_t;

#define FCC_MAX_RANKS 8
#define FCC_MAX_EXPERTS 64
#define FCC_MAX_TABLES 256  /* embedding tables per call */

typedef enum { FCC_BF16 = 0, FCC_F16 = 1, FCC_F32 = 2 } fcc_dtype;

typedef enum {
  FCC_OK = 0,
  FCC_ERR_INVALID = 1,     /* bad argument: null or misaligned pointer, bad size */
  FCC_ERR_UNSUPPORTED = 2, /* valid but not implemented (dtype, algorithm) */
  FCC_ERR_CUDA = 3,        /* a CUDA runtime call failed */
  FCC_ERR_CAPACITY = 4,    /* a receive buffer is too small (MoE cap) */
  FCC_ERR_TIMEOUT = 5,     /* a device-side wait ran out of time */
  FCC_ERR_WORKSPACE = 6    /* caller workspace too small */
} fcc_status;

typedef enum {
  FCC_ALGO_AUTO = 0,       /* chosen per operator and shape (fcc_choose_algo) */
  FCC_ALGO_FUSED = 1,      /* fused GEMM + collective in one persistent kernel */
  FCC_ALGO_UNFUSED = 2,    /* per-rank GEMM to f32 partials, then a reduce/copy kernel */
  FCC_ALGO_INTERDECOM = 3, /* chunks: the GEMM of one chunk overlaps the data movement of
                              another (row chunks; MoE: expert ranges) */
  FCC_ALGO_CE = 4          /* the data between ranks moved by the copy engines
                              (cudaMemcpyAsync), no SMs */
} fcc_algo;

typedef struct {
  fcc_algo algo;
  /* Fused GEMM+ReduceScatter/AllReduce: 1 = ordered tile-owner accumulation
   * (each output tile sums ranks 0..R-1 in order in one accumulator; bitwise
   * repeatable), 0 = push mode (each rank's tile is added into the owner's f32
   * shard with red.global.add.v4.f32; order-free). */
  int deterministic;
  int chunks;              /* InterDecom chunk count; 0 = the cost model */
  int max_ctas;            /* persistent grid size cap; 0 = one CTA per SM */
  int64_t timeout_ns;      /* device wait limit; 0 = 1 s */
  void *workspace;         /* device scratch, or NULL for the internal pool */
  size_t workspace_bytes;
  /* Tensor-core tile shape of the GEMMs: 0 = automatic (a CTA pair when the
   * rows exceed 128 and the 128 x 256 tiles outnumber the CTAs, else 1; the
   * MoE expert GEMM: a CTA pair), 1 = one CTA per 128 x 256 tile, 2 = a CTA pair
   * (cluster of 2, tcgen05 cta_group::2) per 256 x 256 tile.  Any other value
   * is FCC_ERR_INVALID.  Every TMA load lands in the issuing CTA's own shared
   * memory (no multicast loads), so the library may run in processes that
   * drive several GPUs. */
  int cta_pair;
  /* Phase timing, for profiling: NULL (the default), or a device array of
   * 4 uint64 per CTA of the grid (at most the SM count) that the tensor-core
   * GEMM kernels (RS, AR, AG, their unfused GEMMs and the MoE expert GEMM)
   * fill from %globaltimer, for the call's last GEMM launch: [0] ns from the
   * CTA's start to its end, [1] ns its epilogue warps spent on tiles (from an
   * accumulator becoming ready to its last store issued), [2] ns its MMA
   * warp waited for an accumulator the epilogue had not yet handed back (the
   * part of the epilogue not hidden behind the next tile's MMAs; 0 on the
   * second CTA of a pair, which issues no MMAs), [3] tiles it stored. */
  uint64_t *phase_ns;
} fcc_opts;

/* Operator identifiers for fcc_workspace_size. */
typedef enum {
  FCC_OP_GEMM_RS = 0,
  FCC_OP_GEMM_AR = 1,
  FCC_OP_GEMV_AR = 2,
  FCC_OP_AG_GEMM = 3,
  FCC_OP_EMBEDDING_A2A = 4
} fcc_op;

/*
 * GEMM + ReduceScatter (mKernel article, fused kernel list; SC24 abstract).
 *   out_shard[j][i][n] = sum_{r<R} sum_{k<K} A[r][j*M/R + i][k] * B[r][k][n]
 * R in 1..8; A[r]: [M,K] bf16; B[r]: [K,N] bf16; out_shard[j]: [M/R, N] of
 * dtype `out` (FCC_BF16 or FCC_F32).  M % R == 0, K % 8 == 0, N % 8 == 0.
 * Deterministic mode: each output tile sums its k terms (rank after rank)
 * in a fixed order, so results repeat bit for bit and equal fcc_gemm_ar's
 * rows.  When a launch of several rounds of tiles ends with a round of at
 * most half the tiles it could hold, each of those tiles runs as two halves
 * of its k range on two CTA pairs, whose f32 partial sums are then added
 * (still a fixed order); the partials take workspace (fcc_workspace_size).
 * A caller workspace too small for them makes those tiles run as column
 * halves instead, with the tile's whole k range (no error).
 */
fcc_status fcc_gemm_rs(int R, const void *const *A, const void *const *B,
                       void *const *out_shard, int64_t M, int64_t N, int64_t K,
                       fcc_dtype in, fcc_dtype out, const fcc_opts *opts,
                       fcc_stream_t stream);

/*
 * GEMM + AllReduce (mKernel article, fused kernel list).
 *   out[r'] = sum_{r<R} A[r] @ B[r]  for every rank r' (M x N each).
 * Shapes as fcc_gemm_rs (no divisibility of M needed); the same tiling,
 * summation order and workspace use as fcc_gemm_rs.
 */
fcc_status fcc_gemm_ar(int R, const void *const *A, const void *const *B, void *const *out,
                       int64_t M, int64_t N, int64_t K, fcc_dtype in, fcc_dtype out_dtype,
                       const fcc_opts *opts, fcc_stream_t stream);

/*
 * GEMV + AllReduce, the decode shape (SC24 abstract, Transformer operator).
 *   out[r'] = sum_{r<R} A[r] @ B[r] for every rank r'; A[r]: [M,K] with
 *   1 <= M <= 16 tokens; B[r]: [K,N]; out[r']: [M,N] f32 (or bf16).
 * The cross-rank sum is deterministic (fixed order).  Uses workspace.
 */
fcc_status fcc_gemv_ar(int R, const void *const *A, const void *const *B, void *const *out,
                       int64_t M, int64_t N, int64_t K, fcc_dtype in, fcc_dtype out_dtype,
                       const fcc_opts *opts, fcc_stream_t stream);

/*
 * GEMV + AllReduce that allocates nothing.  The pages have no counterpart:
 * this is an addition for callers that cannot call cudaMalloc -- a process
 * whose device memory is already reserved by its own allocator, or a
 * latency-critical path that cannot take cudaMalloc/cudaFree's implicit
 * device synchronisation.  Same arguments and results as fcc_gemv_ar; the
 * caller passes inputs and outputs, and the kernel's scratch (partial sums
 * and arrival tickets) is a 4 MiB static device array inside the library,
 * held on every GPU that loads the library until the process exits.
 *  - Limit: each CTA keeps an M x 512 f32 partial (M x 2 KiB) per group of
 *    512 columns, in the array's 4 MiB less 4 KiB of tickets, so
 *    ceil(N/512) * M <= 2046 (N <= 130,560 for 8 tokens,
 *    65,024 for 16); within that the call uses as many CTAs per column group
 *    as fit in the array (possibly fewer than fcc_gemv_ar uses, which changes
 *    only the f32 summation order).  Beyond it the call returns
 *    FCC_ERR_WORKSPACE and launches nothing.  opts->workspace is ignored;
 *    algo must be AUTO or FUSED (UNFUSED, INTERDECOM and CE give
 *    FCC_ERR_UNSUPPORTED, values outside the enum FCC_ERR_INVALID, as in
 *    fcc_gemv_ar).
 *  - The first call on a device looks up the array's device address and the
 *    SM count (cudaGetSymbolAddress, cudaDeviceGetAttribute) with that device
 *    current; make that first call before any stream capture.
 *  - Every call uses the same array and clears its tickets (cudaMemsetAsync)
 *    first.  Calls that overlap on the GPU (other streams, other threads)
 *    race on the array: serialise them.
 */
fcc_status fcc_gemv_ar_static(int R, const void *const *A, const void *const *B,
                              void *const *out, int64_t M, int64_t N, int64_t K, fcc_dtype in,
                              fcc_dtype out_dtype, const fcc_opts *opts, fcc_stream_t stream);

/*
 * AllGather + GEMM (mKernel article, fused kernel list).
 *   X = [X_shard[0]; ...; X_shard[R-1]]   (each [M/R, K], X is [M, K])
 *   out[r] = X @ B[r]                      ([M, N] per rank, dtype `out_dtype`)
 *   gathered[r] (nullable array, or NULL entries): receives X ([M, K] bf16).
 * opts->algo: FUSED (AUTO) = one kernel whose tiles read their A rows from
 * the owning shard; UNFUSED = a gather kernel into gathered[0] (or
 * workspace), then the per-rank GEMMs; INTERDECOM = the same in row chunks
 * of 256-row tiles, each chunk's gather on a side stream ahead of that
 * chunk's GEMMs (chunk count opts->chunks, else the fcc_interdecom_chunks
 * model with G = the GEMMs, X = the gather); CE = the gather by one
 * cudaMemcpyAsync per shard.  The non-fused forms use workspace of M*K*2
 * bytes when gathered[0] is NULL (fcc_workspace_size).
 */
fcc_status fcc_ag_gemm(int R, const void *const *X_shard, const void *const *B,
                       void *const *out, void *const *gathered, int64_t M, int64_t N,
                       int64_t K, fcc_dtype in, fcc_dtype out_dtype, const fcc_opts *opts,
                       fcc_stream_t stream);

/*
 * MoE Dispatch + GEMM (mKernel article, fused kernel list; SC24 abstract,
 * GEMM + All-to-All for MoE).  R source ranks with T tokens each; E experts,
 * E/R per rank, expert e on rank e/(E/R).
 *   route:    topk_idx[s][t][0..topk) = experts with the largest logits
 *             (ties: lower index first); topk_gate = their softmax probability
 *             over all E experts (not renormalised, not applied below).
 *   dispatch: assignments (s, t, slot) sorted stably by expert; rank d
 *             receives its experts' rows in (expert, s, t, slot) order:
 *             recv_src[d][row] = s*T + t, recv_x[d][row] = X[s][t],
 *             expert_counts[e], send_counts[s*R + d].
 *   GEMM:     recv_y[d][row] = X[s][t] @ W[e]  ([F] per row, dtype out_dtype).
 * X[s]: [T,H] bf16; logits[s]: [T,E] f32, finite; W[e]: [H,F] bf16 (E
 * pointers); recv_x: NULL, or per rank [cap,H] bf16 to receive the
 * dispatched rows.  By default (AUTO) the expert GEMM kernel moves the rows
 * itself, into recv_x or into workspace when it is NULL, one (expert,
 * m tile) unit after another, and its tensor cores read each unit as soon as
 * it is moved.  FCC_ALGO_UNFUSED (the unfused baseline) moves all rows with a
 * separate copy kernel before the GEMM.  FCC_ALGO_INTERDECOM (the chunked
 * baseline) splits the experts into c contiguous ranges (c = opts->chunks,
 * else the fcc_interdecom_chunks model with G = the expert GEMMs, X = the
 * row copy; at most E); each range's rows are copied on a side stream ahead
 * of that range's grouped GEMM, so copy i+1 overlaps GEMM i.  FCC_ALGO_CE
 * (the copy-engine baseline) packs each source rank's kept rows into a send
 * buffer in (expert, token, slot) order (a copy within the rank), reads the
 * (source, expert) run table back to the host (so this form synchronises
 * `stream` before it returns), and moves each run, contiguous on both sides,
 * with one cudaMemcpyAsync on the copy engines, then runs the GEMM.  With
 * opts->algo == FCC_ALGO_FUSED and the sources one [R*T,H] array (X[s] =
 * X[0] + s*T*H elements), the GEMM instead reads each row straight from its
 * source token (TMA gather) and a non-NULL recv_x is filled beside it (slower
 * on sm_103a: the gather is bound by its TMA request rate); FUSED with other
 * sources moves the rows as the default does.  recv_y[d]: [cap,F];
 * recv_src[d]: [cap] int32; topk_idx[s]: [T,topk] int32; topk_gate[s]:
 * [T,topk] f32; expert_counts: [E] int32 device; send_counts: [R*R] int32
 * device.  Rows of a receive buffer past the received count are left
 * untouched.  topk in {1, 2}; R <= E <= 64, E % R == 0; H % 8 == 0;
 * F % 8 == 0.  A rank receiving more than cap rows sets FCC_ERR_CAPACITY in
 * the status word; its rows past cap are dropped (not copied, not multiplied).
 * Index outputs are bit-exact and repeatable (no atomics decide a position).
 * Uses workspace (fcc_moe_workspace_size; with FCC_ALGO_CE in opts it
 * includes the R*T*topk*H*2 bytes of send buffers).
 */
fcc_status fcc_moe_dispatch_gemm(int R, const void *const *X, const float *const *logits,
                                 const void *const *W, int64_t T, int64_t H, int64_t F, int E,
                                 int topk, void *const *recv_x, void *const *recv_y,
                                 int64_t cap, int32_t *const *topk_idx,
                                 float *const *topk_gate, int32_t *expert_counts,
                                 int32_t *send_counts, int32_t *const *recv_src, fcc_dtype in,
                                 fcc_dtype out_dtype, const fcc_opts *opts,
                                 fcc_stream_t stream);

/*
 * MoE combine: the return all-to-all and the gate-weighted top-k sum (SC24
 * abstract, GEMM + All-to-All for MoE: the direction back to the token
 * owners).  For every source rank s and token t:
 *   y[s][t][f] = sum over slots j < topk of topk_gate[s][t][j] * recv_y[d][i][f]
 * where row i of receiving rank d is the row that assignment (s, t, j) was
 * given by the dispatch that produced recv_y (d = topk_idx[s][t][j] / (E/R)),
 * the slots added in order in f32 (so the result is repeatable).  A slot
 * whose row was dropped for capacity adds nothing.  The receive rows are
 * found from recv_src and expert_counts as fcc_moe_dispatch_gemm wrote them:
 * rank d holds its E/R experts' rows in expert order, min(cap, their total)
 * rows in all.
 * recv_y[d]: [cap,F] (in: bf16 or f32); topk_idx[s]: [T,topk] int32;
 * topk_gate[s]: [T,topk] f32; recv_src[d]: [cap] int32; expert_counts: [E]
 * int32 (device); y[s]: [T,F] (out_dtype: bf16 or f32).  topk in {1, 2};
 * R <= E <= 64, E % R == 0; F % 8 == 0.  Uses workspace
 * (fcc_moe_combine_workspace_size).
 */
fcc_status fcc_moe_combine(int R, const void *const *recv_y, int64_t cap, int64_t T, int64_t F,
                           int E, int topk, const int32_t *const *topk_idx,
                           const float *const *topk_gate, const int32_t *const *recv_src,
                           const int32_t *expert_counts, void *const *y, fcc_dtype in,
                           fcc_dtype out_dtype, const fcc_opts *opts, fcc_stream_t stream);

/*
 * Embedding + All-to-All (SC24 abstract: the embedding + All-to-All operator
 * for DLRM).  ntables embedding tables [V, D] (table t owned by rank
 * t / (ntables / R)); R ranks with Bl samples each (global sample g lives on
 * rank g / Bl).  Bag (t, g) is the index list
 * indices[t][offsets[t][g] .. offsets[t][g + 1]) into table t; its pooled
 * vector is the sum of those rows (f32, then stored in out_dtype; an empty
 * bag gives zeros).  The all-to-all delivers it to the sample's rank:
 *   out[g / Bl][g % Bl][t][:] = pooled vector of bag (t, g)
 * tables[t]: [V, D] bf16; offsets[t]: [R*Bl + 1] int32, non-decreasing;
 * indices[t]: [offsets[t][R*Bl]] int32 in [0, V); out[r]: [Bl, ntables, D]
 * (bf16 or f32).  R <= 8, ntables % R == 0, ntables <= FCC_MAX_TABLES,
 * D % 8 == 0.  opts->algo: FUSED (AUTO) = one kernel pools each bag and
 * stores it straight into its sample's rank buffer; UNFUSED = each table's
 * pooled vectors into a [ntables, R*Bl, D] workspace, then a kernel moves
 * them to the sample ranks; CE = the same workspace moved by copy-engine 2-D
 * copies (one per table and rank).  A negative offset step or an index
 * outside [0, V) is not read: the bag skips it and FCC_ERR_INVALID is
 * recorded in the status word.  Within a call the result is repeatable (a
 * fixed summation order).  Uses workspace for UNFUSED / CE
 * (fcc_embedding_workspace_size).
 */
fcc_status fcc_embedding_a2a(int R, int ntables, const void *const *tables, int64_t V,
                             int64_t D, int64_t Bl, const int32_t *const *offsets,
                             const int32_t *const *indices, void *const *out, fcc_dtype in,
                             fcc_dtype out_dtype, const fcc_opts *opts, fcc_stream_t stream);
size_t fcc_embedding_workspace_size(int R, int ntables, int64_t D, int64_t Bl,
                                    fcc_dtype out_dtype, const fcc_opts *opts);

/*
 * Ring attention (the mKernel article's fused kernel list: Ring Attention).
 * The sequence is split over R ranks, S positions each (rank r's row t is
 * global position r*S + t); every rank's queries attend to the keys and
 * values of all shards, which the ring brings round (here: each CTA reads
 * the blocks of every shard in ring order, its own shard first):
 *   O_r[t][h] = sum_j softmax_j(Q_r[t][h] . K[j][h] / sqrt(d)) V[j][h]
 * over all global positions j (causal != 0: only j <= r*S + t).
 * Q[r], K[r], V[r]: [S, H, d] bf16; O[r]: [S, H, d] (bf16 or f32).  d = 128
 * (others: FCC_ERR_UNSUPPORTED).  Scores, softmax and sums in f32; the
 * probabilities (relative to a running row maximum) enter the P V product as
 * bf16.  Repeatable (a fixed order).  No workspace.
 */
fcc_status fcc_ring_attention(int R, const void *const *Q, const void *const *K,
                              const void *const *V, void *const *O, int64_t S, int H, int64_t d,
                              int causal, fcc_dtype in, fcc_dtype out_dtype,
                              const fcc_opts *opts, fcc_stream_t stream);

/* Scratch bytes a call needs (for opts->workspace); 0 if none. */
size_t fcc_workspace_size(fcc_op op, int R, int64_t M, int64_t N, int64_t K,
                          const fcc_opts *opts);
size_t fcc_moe_workspace_size(int R, int64_t T, int64_t H, int64_t F, int E, int topk,
                              int64_t cap, const fcc_opts *opts);
size_t fcc_moe_combine_workspace_size(int R, int64_t T, int topk);

/*
 * Synchronises `stream`, then returns and clears the device status word of
 * the current device (FCC_OK if no device-side error was recorded).
 */
fcc_status fcc_stream_status(fcc_stream_t stream);

/* Static description of a status code. */
const char *fcc_status_string(fcc_status s);

/*
 * The algorithm FCC_ALGO_AUTO runs for a call (the strategy selector, after
 * Compass's unified framework of operator variants: "Compass: Dissecting
 * Communication and Computation Operators for Efficient LLM Training",
 * abstract), from measurements on GB300: FCC_ALGO_FUSED for the GEMM +
 * ReduceScatter / AllReduce and AllGather + GEMM (fastest at every shape
 * measured); for the GEMV + AllReduce, FCC_ALGO_UNFUSED when the fused grid
 * would split the rank-and-K range 16 or more ways (few 512-column groups:
 * its final serial sum of the splits then costs more than the plain GEMM +
 * reduce), else FCC_ALGO_FUSED; for the embedding + All-to-All,
 * FCC_ALGO_FUSED (1133-1140 us on 8 ranks x 64 tables of 65536 x 128, 2048
 * samples a rank, bags of 32, against 1304-1308 us for pooling table by table
 * into a staging buffer and then the exchange).  sms: SMs to plan for (0 =
 * the current device's, 152 without one); max_ctas as in fcc_opts.
 * Host-only.
 */
fcc_algo fcc_choose_algo(fcc_op op, int R, int64_t M, int64_t N, int64_t K, int sms,
                         int max_ctas);

/*
 * InterDecom chunk-count model ("Compass: Dissecting Communication and
 * Computation Operators for Efficient LLM Training", abstract: a model that
 * derives the optimal decomposition degree; its formula is not given there).
 * Two-stage pipeline, c chunks, per-chunk overhead alpha:
 *   T(c) = max(G, X) + min(G, X) / c + c * alpha
 * minimised at c* = sqrt(min(G, X) / alpha), rounded to the better integer
 * neighbour and clamped to [1, max_chunks].  G = one-shot GEMM time, X =
 * one-shot collective time (any consistent unit).
 */
int fcc_interdecom_chunks(double G, double X, double alpha, int max_chunks);
double fcc_interdecom_time(double G, double X, double alpha, int chunks);

/*
 * Test support: launches one kernel whose bounded wait on a barrier that
 * nothing completes runs out after timeout_ns; the kernel then records
 * FCC_ERR_TIMEOUT in the status word and returns, leaving the context usable.
 * fcc_stream_status() afterwards returns FCC_ERR_TIMEOUT.
 */
fcc_status fcc_test_wait_timeout(int64_t timeout_ns, fcc_stream_t stream);

/*
 * Test support: launches the MoE grouped expert GEMM kernel (the in-kernel
 * staging form of fcc_moe_dispatch_gemm) on a one-tile table whose unit row
 * counter nothing raises, so its TMA producers' bounded wait for the unit's
 * rows runs out after timeout_ns; the kernel records FCC_ERR_TIMEOUT and
 * returns, leaving the context usable.  Uses the internal workspace pool.
 */
fcc_status fcc_test_grouped_wait_timeout(int64_t timeout_ns, fcc_stream_t stream);

/*
 * Test support: launches the fused GEMM + ReduceScatter kernel on a small
 * problem (1 rank, 384 x 256 x 128, on two single CTAs) whose short last
 * round runs as two K halves, with the second half waiting for a flag value
 * the first never writes, so that bounded wait runs out after timeout_ns;
 * the kernel records FCC_ERR_TIMEOUT, stores nothing for that tile and
 * returns, leaving the context usable.  Uses the internal workspace pool.
 */
fcc_status fcc_test_ksplit_wait_timeout(int64_t timeout_ns, fcc_stream_t stream);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t fcc_launch_count(void);

/* Library version, "major.minor.patch". */
const char *fcc_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FCC_H_ */
