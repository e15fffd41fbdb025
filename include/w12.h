/*
 * w12.h -- C ABI of the GB300-native W12 speculative-decoding verify path.
 *
 * The verify pass of a speculative decoder reads every target weight to score
 * a small block (or tree) of drafted tokens per request (SpecPilot paper
 * digest, summary paragraph). Weights are stored in W12, a lossless 12-bit
 * layout: BF16 is split into three 4-bit planes that the GEMM restores
 * bitwise in registers (SpecPilot digest, "Reasons" bullet 2). Acceptance is
 * greedy: a drafted token is kept iff it equals the target's argmax at the
 * preceding position (SpecPilot digest, "Risks" bullet 3); draft trees are
 * causal, each token conditioned on its root-to-node path (JetSpec article,
 * "Technical architecture").
 *
 * W12 layout used by this library (the pages fix only "three 4-bit planes,
 * restored bitwise"; the mapping below is this library's definition):
 *   - rows n of W[N, K] (out x in, bf16) are cut into groups of 128 K values;
 *   - per group, ebase = max(emax - 15, 0), emax = the largest biased exponent
 *     among the group's finite nonzero normal values (0 if none);
 *   - a normal finite value with exponent e > ebase is coded as
 *     code12 = s<<11 | (e-ebase)<<7 | m; anything else (zeros, subnormals,
 *     magnitudes below the 15-binade window, Inf, NaN) is coded 0 and listed
 *     in the exception CSR with its exact 16 bits;
 *   - plane p (p = 0, 1, 2) stores nibble p of code12, bytes [N, K/2]; in each
 *     row the elements 8q..8q+7 fill bytes 4q..4q+3: byte 4q+i holds element
 *     8q+i in its low nibble and element 8q+4+i in its high nibble;
 *   - ebase is a byte array [K/128, N] (group-major);
 *   - exceptions: blocks of 128 rows x 128 columns, u = (n/128)*(K/128)+k/128;
 *     exc_off[u] .. exc_off[u+1] index exc_ent; an entry is
 *     (n%128)<<23 | (k%128)<<16 | bf16 bits, ascending within a block.
 *
 * Conventions for every entry point:
 *   - Pointers named in the argument lists are DEVICE pointers into memory the
 *     caller owns (e.g. allocated by PyTorch), unless the comment says "host".
 *     The library never allocates and never frees memory.
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream). Entry points return once the work is
 *     enqueued; only the *_query and w12_pack calls synchronise the stream.
 *   - Return value: W12_OK or an error code; argument and shape errors are
 *     detected on the host before anything is enqueued.
 *   - `dev_status` (nullable device int32): kernels that detect an error at
 *     run time (a bounded wait that expired, a malformed tree) store the first
 *     such W12_ERR_* code there; the caller reads it after synchronising.
 *     The word is never cleared by the library.
 *   - `ws` / `ws_bytes`: caller-owned device workspace of at least the size
 *     the matching *_ws_bytes function returns, ZERO-FILLED before its first
 *     use; the library leaves it zeroed after every successful call, so it can
 *     be reused. After an error status, zero it again. Calls that share one
 *     workspace must not overlap in time (same stream, or synchronised).
 *   - Shapes: N % 128 == 0, K % 128 == 0, 1 <= M <= 256 rows.
 */
#ifndef W12_H
#define W12_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
  W12_OK = 0,
  W12_ERR_ARG = 1,        /* null pointer, bad enum, misaligned pointer      */
  W12_ERR_SHAPE = 2,      /* K or N not a multiple of 128, M outside 1..256  */
  W12_ERR_WORKSPACE = 3,  /* workspace or exception capacity too small       */
  W12_ERR_BAD_TREE = 4,   /* parents[0] != -1 or parents[i] not in [0, i)    */
  W12_ERR_CORRUPT = 5,    /* packed weights fail a consistency check         */
  W12_ERR_TIMEOUT = 6,    /* a device-side bounded wait expired              */
  W12_ERR_CUDA = 7,       /* a CUDA runtime call failed                      */
  W12_ERR_UNSUPPORTED = 8 /* no sm_103a device, or the shape needs a feature
                             this build does not have                        */
};

/* W12-packed weight matrix: plain data holding device pointers.
 *   p0, p1, p2 : N*K/2 bytes each, 16-byte aligned
 *   ebase      : (K/128)*N bytes
 *   exc_off    : (N/128)*(K/128) + 1 uint32
 *   exc_ent    : n_exc uint32 (capacity when passed to w12_pack) */
typedef struct w12_weights {
  int64_t N, K;
  uint8_t* p0;
  uint8_t* p1;
  uint8_t* p2;
  uint8_t* ebase;
  uint32_t* exc_off;
  uint32_t* exc_ent;
  int64_t n_exc;
} w12_weights;

/* Byte sizes of the buffers of a packed N x K matrix (host struct). */
typedef struct w12_sizes {
  int64_t plane_bytes;    /* per plane: N*K/2                     */
  int64_t ebase_bytes;    /* (K/128)*N                            */
  int64_t exc_off_count;  /* (N/128)*(K/128) + 1                  */
  int64_t n_exc;          /* exception entries of this matrix     */
  int64_t total_bytes;    /* 1.5NK + NK/128 + 4*(U+1) + 4*n_exc   */
} w12_sizes;

/* Human-readable name of a status code (static string, never NULL). */
const char* w12_status_string(int status);

/* Library ABI version (major*100 + minor). */
int w12_version(void);

/* --- W12 pack / unpack (SpecPilot digest, "Reasons" bullet 2) ----------- */

/* Workspace for w12_pack_query: (N/128)*(K/128)+1 uint32 counters. */
size_t w12_pack_ws_bytes(int64_t N, int64_t K);

/* Count the exceptions of bf16 W[N, K] (row-major) and fill *out (host).
 * Synchronises `stream`. */
int w12_pack_query(const uint16_t* W, int64_t N, int64_t K, w12_sizes* out,
                   void* ws, size_t ws_bytes, void* stream);

/* Pack bf16 W[N, K] into *dst (host struct; its buffers sized per
 * w12_pack_query, dst->n_exc = capacity of dst->exc_ent). On success
 * dst->n_exc is NOT modified; the exact count is exc_off[U]. Returns
 * W12_ERR_WORKSPACE if the exceptions exceed the capacity. Synchronises. */
int w12_pack(const uint16_t* W, int64_t N, int64_t K, const w12_weights* dst, void* stream);

/* Restore bf16 W_out[N, K] bit-exactly from a packed matrix. A corrupt
 * exception CSR (offsets that decrease, an offset past n_exc, or an entry
 * whose row field is 128 or more) stores W12_ERR_CORRUPT in dev_status
 * (nullable); the affected block's exceptions are then not applied, and no
 * store ever lands outside W_out. */
int w12_unpack(const w12_weights* src, uint16_t* W_out, int32_t* dev_status, void* stream);

/* --- Verify GEMM (SpecPilot digest, summary; "Reasons" bullet 2) -------- */

/* Workspace bytes for w12_gemm / w12_gemm_bf16_ref at this shape. */
size_t w12_gemm_ws_bytes(int64_t M, int64_t N, int64_t K);

/* Y[M, N] (fp32, row-major) = X[M, K] (bf16, row-major) * W^T, W restored
 * from its three planes inside the kernel. X must be 16-byte aligned. A
 * corrupt exception CSR (as for w12_unpack) stores W12_ERR_CORRUPT in
 * dev_status; the output is then unspecified, and no access leaves the
 * buffers the descriptor names. */
int w12_gemm(const uint16_t* X, int64_t M, const w12_weights* W, float* Y,
             void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Same product as w12_gemm without a caller workspace, for callers that
 * cannot allocate device memory: code embedded in a host application that
 * owns every device allocation and exposes no allocator, and latency-critical
 * loops that may not call cudaMalloc/cudaFree (or a framework allocator)
 * while they run. The pages have no counterpart to this entry point.
 * The split-K scratch is a fixed array of 3,162,112 bytes that the library
 * holds in device memory on every GPU where it is loaded, until the process
 * exits. It serves M <= 16 rows, N <= 524288 (4096 tiles of 128), and GPUs
 * with up to 192 SMs; larger shapes return W12_ERR_WORKSPACE (use w12_gemm).
 * The first call in each CUDA context (the device's primary context, or one
 * the caller created) looks up the array's device address in that context,
 * with it current; make that first call before any stream capture. Every
 * call clears the tile counters it uses and allocates nothing. All calls
 * share the one array: calls that overlap on the GPU (other streams, or
 * several host threads) race and corrupt each other's results; serialise
 * them. X, Y, dev_status and stream are as for w12_gemm. */
int w12_gemm_noalloc(const uint16_t* X, int64_t M, const w12_weights* W, float* Y,
                     int32_t* dev_status, void* stream);

/* Same product with W given as plain bf16 [N, K] (the in-tree BF16 baseline
 * that shows what the 12/16 byte saving is worth). */
int w12_gemm_bf16_ref(const uint16_t* X, int64_t M, const uint16_t* W, int64_t N, int64_t K,
                      float* Y, void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* --- Grouped verify GEMMs in one launch -------------------------------- */
/* The verify pass reads every target weight each step (SpecPilot digest,
 * summary); a dense layer has several such GEMMs at the same M. A grouped
 * launch runs up to 4 of them in one persistent kernel (one ramp-up and one
 * tail for the group instead of one per GEMM): the SMs are split over the
 * problems in proportion to their 128x128 units, and each problem's units are
 * split evenly over its SMs. With a SwiGLU link, problem `to` takes
 * as X the gated activation of problem `from`'s output, computed inside the
 * launch: act[m, j] = bf16(silu(Y_from[m, j]) * Y_from[m, N_from/2 + j]),
 * silu(g) = g / (1 + exp(-g)), rounded to nearest even. The pages give no
 * MLP activation; this is the gated SiLU of dense decoder layers, with the
 * gate in the first half of the fused gate/up output. The launch then runs
 * in three phases, the SMs split anew in each: the source, the other
 * problems, the target; each of the target's k-blocks starts once that block
 * of act is written.
 *
 * problems: X [M, K] bf16 row-major (16-byte aligned; unused for the link
 * target), weights (W for w12_gemm_grouped; Wbf16 with N, K for the bf16
 * baseline), Y [M, N] fp32 output. All problems share M (1..256). The link
 * needs N_from % 256 == 0 and K_to == N_from / 2; act is caller-owned
 * [M, N_from/2] bf16, 16-byte aligned, and is overwritten. Y_from is written
 * as well. The workspace must be zero-filled before its first use; the
 * library leaves it ready for the next call after a W12_OK call (zero it
 * again after any error). Grouped calls that share a workspace must not
 * overlap on the GPU. Errors: W12_ERR_ARG, W12_ERR_SHAPE (a shape rule, or
 * more than 1023 units per SM), W12_ERR_WORKSPACE, W12_ERR_UNSUPPORTED,
 * W12_ERR_CUDA; W12_ERR_TIMEOUT in dev_status if a wait gives up. */
typedef struct w12_problem {
  const uint16_t* X;
  const w12_weights* W;
  const uint16_t* Wbf16;
  int64_t N, K;
  float* Y;
} w12_problem;

typedef struct w12_swiglu {
  int from, to;
  uint16_t* act;
} w12_swiglu;

/* Workspace bytes for a grouped call (0 if the arguments are invalid).
 * probs[i].W decides the mode: W12 if probs[0].W is set, else bf16. */
size_t w12_gemm_grouped_ws_bytes(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link);

int w12_gemm_grouped(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link,
                     void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* The same grouped launch over plain bf16 weights (in-tree baseline). */
int w12_gemm_grouped_bf16_ref(const w12_problem* probs, int n, int64_t M, const w12_swiglu* link,
                              void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* --- Commit of the accepted path ---------------------------------------- */
/* The step after acceptance (SpecPilot digest, "Reasons" bullet 2: tree
 * verification for targets with recurrent layers; JetSpec article,
 * "Technical architecture": each draft token is conditioned on its
 * root-to-node path). The verify pass wrote one row per draft node into
 * each cache: node i of request b at position prefix_len[b] + i. The pages do
 * not describe the cache; this library's reading is a row-major array
 * [B, S_max, row_bytes] per cache (one per layer and per K or V, any element
 * type; row_bytes a multiple of 16, base 16-byte aligned).
 *
 * w12_kv_commit moves, for every cache and request, row prefix_len[b] +
 * path[b, k] to row prefix_len[b] + k for k < path_len[b], in place, and
 * writes new_len[b] = prefix_len[b] + path_len[b] (new_len may be NULL).
 * path [B, path_stride] is root-first with strictly increasing node indices
 * (the tree verify output is such a path; a greedy block's accepted prefix is
 * 0, 1, ..., L, which moves nothing). A request whose path is invalid (empty,
 * longer than path_stride, not increasing, or reaching past S_max) is left
 * unchanged, gets new_len = prefix_len, and sets W12_ERR_BAD_TREE in
 * dev_status. caches is a HOST array of n_caches device pointers; prefix_len,
 * path, path_len and new_len are device arrays. Rows past the new length keep
 * whatever they held. Errors: W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_CUDA. */
int w12_kv_commit(void* const* caches, int n_caches, int B, int64_t S_max, int64_t row_bytes,
                  const int32_t* prefix_len, const int32_t* path, int path_stride, const int32_t* path_len,
                  int32_t* new_len, int32_t* dev_status, void* stream);

/* Recurrent state of the accepted node: out[b] = states[b, node] with node =
 * path[b, path_len[b] - 1], states [B, T, row_bytes] (one state per draft
 * node, written by the verify pass), out [B, row_bytes]. An invalid path sets
 * W12_ERR_BAD_TREE in dev_status and leaves out[b] unchanged. */
int w12_state_select(const void* states, int B, int T, int64_t row_bytes, const int32_t* path, int path_stride,
                     const int32_t* path_len, void* out, int32_t* dev_status, void* stream);

/* --- Tree-masked verify attention ---------------------------------------- */
/* The attention half of the target's verify pass over a causal draft tree
 * (JetSpec article, "Technical architecture": every draft token is
 * conditioned on the path that leads to it; SpecPilot digest, "Reasons"
 * bullet 2: tree verification; a block of T drafted tokens is the chain tree
 * parents[i] = i - 1). The pages give no attention details; this library's
 * reading:
 *   O[b, t, h, :] = sum_j softmax_j(scale * Q[b, t, h, :] . K[b, j, h / G, :])
 *                   * V[b, j, h / G, :],   G = Hq / Hkv,
 * over the keys j < prefix_len[b] and j = prefix_len[b] + i for every node i
 * on the path root -> t (t included). Layouts (all bf16, contiguous, 16-byte
 * aligned device memory): Q and O [B, T, Hq, head_dim], K_cache and V_cache
 * [B, S_max, Hkv, head_dim], node i's key/value at position prefix_len[b] + i
 * (written by the verify pass before this call). parents [B, T] int32
 * (parents[b, 0] = -1, 0 <= parents[b, i] < i), prefix_len [B] int32, both
 * device arrays. head_dim must be 128; 1 <= T <= 128; Hq a multiple of Hkv.
 * max_kv_len (host) bounds prefix_len[b] + T over the requests, T <= max_kv_len
 * <= S_max; the work split is planned for it. scale > 0. Cache rows at or past
 * prefix_len[b] + T are never used (they may hold anything). Computes in fp32
 * with P rounded to bf16 for the P.V product and O rounded to bf16.
 * Device-side errors in dev_status: W12_ERR_BAD_TREE (malformed parents; that
 * request's outputs are unspecified), W12_ERR_ARG (prefix_len[b] < 0 or
 * prefix_len[b] + T > max_kv_len; the request is computed with its prefix
 * clamped into range), W12_ERR_TIMEOUT (a bounded wait gave up; outputs
 * unspecified). Returns W12_ERR_ARG, W12_ERR_SHAPE, W12_ERR_WORKSPACE,
 * W12_ERR_UNSUPPORTED or W12_ERR_CUDA. The workspace is at least
 * w12_tree_attention_ws_bytes(...) bytes, which is 0 for a shape the call
 * rejects. It holds the key splits' partial results and one arrival count per
 * (request, kv head, row tile): zero-fill it before its first use; a call
 * that ends with dev_status W12_OK leaves the counts at zero, so the same
 * workspace serves the next call. After any error status, zero it again.
 * Calls that share one workspace must be ordered on one stream. */
size_t w12_tree_attention_ws_bytes(int B, int T, int Hq, int Hkv, int64_t max_kv_len);

int w12_tree_attention(const uint16_t* Q, const uint16_t* K_cache, const uint16_t* V_cache, int B, int T, int Hq,
                       int Hkv, int head_dim, int64_t S_max, int64_t max_kv_len, const int32_t* prefix_len,
                       const int32_t* parents, float scale, uint16_t* O, void* ws, size_t ws_bytes,
                       int32_t* dev_status, void* stream);

/* --- Greedy block verification (SpecPilot digest, "Risks" bullet 3) ----- */

/* Workspace bytes for the verify entry points with M = B*rows verified rows
 * over a vocabulary of V (V % 128 == 0 for the fused forms). */
size_t w12_verify_ws_bytes(int64_t M, int64_t V);

/* logits [B*T_rows, V] fp32. Row j of request b is the target's prediction
 * for draft token j. accept_len[b] = longest L <= T with
 * draft[b, j] == argmax(row b*T_rows + j) for all j < L; bonus[b] =
 * argmax(row b*T_rows + L) if L < T_rows, else -1. Argmax ties resolve to the
 * lowest index. T_rows is T or T+1. argmax_out [B*T_rows] is optional. */
int w12_verify_greedy(const float* logits, int64_t V, const int32_t* draft, int B, int T, int T_rows,
                      int32_t* accept_len, int32_t* bonus, int32_t* argmax_out,
                      void* ws, size_t ws_bytes, int32_t* dev_status, void* stream);

/* Same, with the logits computed on the fly by the W12 LM head:
 * H [B*T_rows, K] bf16 hidden states, head = W12 [V, K]. The logits are never
 * written to memory; each 128-row vocabulary tile reduces to a per-row
 * (max, index) pair inside the GEMM epilogue. */
int w12_verify_greedy_fused(const uint16_t* H, const w12_weights* head, const int32_t* draft,
                            int B, int T, int T_rows, int32_t* accept_len, int32_t* bonus,
                            int32_t* argmax_out, void* ws, size_t ws_bytes, int32_t* dev_status,
                            void* stream);

/* --- Tree verification (JetSpec article, "Technical architecture";
 *     SpecPilot digest, "Reasons" bullet 2) ------------------------------- */

/* B trees of T nodes; node 0 of each tree is the committed anchor, parents
 * [B, T] with parents[b, 0] = -1 and 0 <= parents[b, i] < i. Row b*T + p of
 * logits [B*T, V] is the target's prediction after the path root..p. Node
 * i > 0 is accepted iff its parent is accepted and draft[b, i] equals the
 * argmax of its parent's row. Output per tree: the accepted node of greatest
 * depth (lowest index among equals): path [B, T] root-first (-1 padded),
 * path_len [B] = depth + 1, accept_len [B] = depth, bonus [B] = argmax of
 * that node's row. A malformed tree sets W12_ERR_BAD_TREE in dev_status and
 * -1 in its outputs. argmax_out [B*T] is optional. */
int w12_verify_tree(const float* logits, int64_t V, const int32_t* parents, const int32_t* draft,
                    int B, int T, int32_t* path, int32_t* path_len, int32_t* accept_len,
                    int32_t* bonus, int32_t* argmax_out, void* ws, size_t ws_bytes,
                    int32_t* dev_status, void* stream);

/* Same, with the fused W12 LM head over H [B*T, K]. */
int w12_verify_tree_fused(const uint16_t* H, const w12_weights* head, const int32_t* parents,
                          const int32_t* draft, int B, int T, int32_t* path, int32_t* path_len,
                          int32_t* accept_len, int32_t* bonus, int32_t* argmax_out, void* ws,
                          size_t ws_bytes, int32_t* dev_status, void* stream);

/* --- Diagnostics -------------------------------------------------------- */

/* Launch a kernel that waits on a barrier nothing arrives at, with a bound of
 * `limit_us` microseconds; it must store W12_ERR_TIMEOUT in dev_status and
 * return (no fault, no hang). Used by the failure-detection tests. */
int w12_selftest_timeout(int32_t* dev_status, int limit_us, void* stream);

/* Bound (microseconds) used by every device-side wait of later launches;
 * default 2000000. Values below 1 are rejected. */
int w12_set_wait_limit_us(int64_t limit_us);

/* Copy `bytes` bytes from src to dst on `stream` with a kernel rather than a
 * copy-engine transfer, for the host path of a step (inputs in, results out).
 * dst and src are device memory or page-locked host memory (cudaHostAlloc or
 * cudaHostRegister; the device reads and writes it in place through unified
 * addressing), both 16-byte aligned, not overlapping. With launch overlap on
 * (below) the next kernel on the stream may start while the copy runs (a GEMM
 * then requests its first weight tiles meanwhile), and the copy itself waits
 * for the previous kernel before it reads or writes. bytes == 0 launches
 * nothing. Errors: W12_ERR_ARG (null, misaligned or overlapping pointers, or
 * memory the device cannot address), W12_ERR_UNSUPPORTED, W12_ERR_CUDA. */
int w12_copy(void* dst, const void* src, size_t bytes, void* stream);

/* Launch overlap (programmatic dependent launch), on by default: a GEMM or
 * verify launch may start while the previous kernel on its stream is still
 * running. Before that kernel completes it only reads the packed weights
 * (planes, ebase, exception CSR); it reads X/H/logits/drafts and writes any
 * output or workspace only after waiting for it. So packed weights must not
 * be written by the kernel launched immediately before on the same stream
 * (a copy-engine transfer or an event in between is fine). Pass 0 to launch
 * with ordinary stream ordering. Returns W12_OK. */
int w12_set_overlap(int enable);

#ifdef __cplusplus
}
#endif

#endif /* W12_H */
