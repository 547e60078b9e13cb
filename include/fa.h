/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention-2 backward library.
 *
 * The library computes the backward pass of scaled-dot-product attention
 *
 *     S = scale * Q K^T,   P = softmax(S) row-wise,   O = P V
 *
 * without ever storing an N x N matrix: S and P are recomputed tile by tile
 * on chip from Q, K and the per-row logsumexp L saved by the forward pass
 * ("CUDA 算子工程" ch.16 "FA2 反向", §16.2 loop order and §16.4 role of LSE).
 *
 * A backward pass is three calls on one stream:
 *     fa_bwd_preprocess   D = rowsum(O * dO), zero the fp32 dQ accumulator
 *     fa_bwd              dK, dV written once per key block; dQ partials
 *                         reduced into the fp32 accumulator
 *     fa_convert_dq       dQ = scale * accumulator, cast to the output dtype
 * and fa_fwd produces O and L for it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Q, O, dO, dQ are [B, H, N, d] and K, V, dK, dV [B, H, N_k, d] tensors of
 *    `dtype` with the last dimension contiguous and element strides
 *    (stride_b, stride_h, stride_n), respectively (kstride_b, kstride_h,
 *    kstride_n); N_k = 0 in fa_problem means N_k = N with one set of strides
 *    for all eight tensors (self-attention, the case the pages describe).
 *  - L and D are dense [B, H, N] float32 arrays (row-major, no padding).
 *  - The dQ accumulator is a float32 array of fa_dq_accum_elems() elements in
 *    a tile-blocked layout (below).  It belongs to the caller like every
 *    other buffer: the library never allocates device memory and keeps only
 *    one 4-byte device status word per device.
 *  - All pointers are device pointers that the current CUDA device can
 *    access, 16-byte aligned; every byte stride (stride * element size) must
 *    be a multiple of 16.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  All calls are asynchronous on that stream.
 *  - Arguments are validated on the host before anything is launched; a
 *    rejected call launches nothing and returns FA_ERR_INVALID_ARG or
 *    FA_ERR_UNSUPPORTED.  A failed launch returns FA_ERR_CUDA.  Errors found
 *    on the device (a bounded wait that ran out, a failed self check) never
 *    trap: the kernel records a code in the device status word and returns;
 *    read it with fa_get_device_status().
 *  - Results are not bitwise reproducible from run to run: dQ partial sums
 *    reach the accumulator in whatever order the hardware completes its
 *    reductions (the FA2 default; ch.16 §16.3 notes deterministic=False).
 *
 * Supported problems (N is the number of query rows, N_k of key rows; see
 * fa_problem): dtype FA_BF16 with d in {32, 64, 96, 128, 256} (tcgen05
 * tensor-core kernels; at d = 256 the backward splits each key block over
 * two CTAs by output columns, since the dK and dV accumulators of one block
 * would fill tensor memory); dtype FA_FP32 with d in {16, 32, 64, 96, 128,
 * 256} (exact fp32 FFMA kernels, no TF32).  N >= 1, N_k >= 0, B >= 1,
 * H >= 1, N, N_k <= 2^24, B*H <= 2^24, and B*H*ceil(max(N, N_k)/32) < 2^30
 * (the kernels' 1-D grids).
 * Other d return FA_ERR_UNSUPPORTED.
 *
 * dQ accumulator layout
 * ---------------------
 * Query rows are grouped into tiles of 128 rows; the last tile of a head is
 * padded to 128 rows.  Inside a tile the rows form 4 quarters of 32 and the
 * columns blocks of 16; each (quarter, block) pair is a 2 KB unit laid out
 * [4 column groups of 4][32 rows][4 columns].  Element (b, h, n, c) lives at
 * float index
 *
 *   ((((b*H + h) * T + n/128) * 4 + (n%128)/32) * (d/16) + c/16) * 512
 *     + ((c%16)/4) * 128 + (n%32) * 4 + c%4
 *
 * with T = ceil(N/128).  One unit is what the tensor-core kernel stages in
 * shared memory and adds into the accumulator with one bulk reduction.
 * Padding rows receive only zero contributions.  With FA_FLAG_DETERMINISTIC
 * the accumulator is a sequence of such arrays (slices), one per key block,
 * slice k at float offset k * B*H*T*128*d.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or stride   */
  FA_ERR_UNSUPPORTED = 2,  /* valid problem outside the supported set        */
  FA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed           */
  FA_ERR_TIMEOUT = 4,      /* device: a bounded wait ran out                 */
  FA_ERR_DEVICE = 5        /* device: a kernel self check failed             */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/* fa_problem.flags bits. */
typedef enum {
  /* Bitwise reproducible dQ (ch.16 §16.3 and §16.8 item 4: extra memory buys
   * a fixed summation order).  The accumulator then holds one slice per key
   * block; the backward writes each key block's dQ contribution into its own
   * slice instead of adding it, and fa_convert_dq sums the slices in
   * increasing key-block order. */
  FA_FLAG_DETERMINISTIC = 1
} fa_flags;

/* Shapes: Q, O, dO, dQ are [B, H, N, d] with strides (stride_b, stride_h,
 * stride_n); K, V, dK, dV are [B, H, N_k, d] with strides (kstride_b,
 * kstride_h, kstride_n); L and D are dense [B, H, N] float32.  N_k = 0 means
 * self-attention, N_k = N with the K/V strides equal to the Q strides (the
 * kstride fields are then ignored).
 *
 * Causal mask (N_k != N is not covered by the source pages, which show only
 * N_q == N_k): aligned bottom-right, key j is visible to query i iff
 * j <= i + (N_k - N); at N_k == N this is the pages' j <= i.  A query that
 * sees no key (only possible when N > N_k) gets O = 0, L = +inf and zero
 * gradients. */
typedef struct {
  int32_t B, H, N, d;
  float scale;      /* softmax scale, normally 1/sqrt(d) */
  int32_t causal;   /* 1: key j visible to query i iff j <= i + N_k - N */
  int32_t dtype;    /* fa_dtype of Q, K, V, O, dO, dQ, dK, dV */
  int32_t flags;    /* fa_flags bits (0: default mode); other bits must be 0 */
  int64_t stride_b, stride_h, stride_n; /* element strides of Q-shaped tensors; d is contiguous */
  int32_t N_k;      /* key/value rows; 0: equal to N (self-attention) */
  int32_t reserved; /* must be 0 */
  int64_t kstride_b, kstride_h, kstride_n; /* element strides of K-shaped tensors (N_k > 0) */
} fa_problem;

/* Number of float32 elements of the dQ accumulator for problem p, or 0 if p
 * is NULL or invalid: B * H * ceil(N/128) * 128 * d, times the number of key
 * blocks with FA_FLAG_DETERMINISTIC: ceil(N_k/128) for bf16 (tensor-core
 * backward), ceil(N_k/64) for fp32 (CUDA-core backward), ceil(N_k/32) for
 * fp32 at d = 256. */
size_t fa_dq_accum_elems(const fa_problem* p);

/* Forward pass, companion of the backward: O = softmax(scale Q K^T) V and
 * L = logsumexp of each row of scale Q K^T (natural log).  Online softmax
 * over key blocks with running max m, sum l and rescale alpha = exp(m - m')
 * (1point3acres FlashAttention write-up, online-softmax paragraphs; ch.16
 * §16.4 L = m + log l).  Reads Q, K, V; writes O (dtype) and L (float32). */
fa_status fa_fwd(const fa_problem* p, const void* Q, const void* K, const void* V,
                 void* O, float* L, void* stream);

/* Backward preprocess (ch.16 §16.8 item 1; identity of §16.1):
 * D[b,h,n] = sum_c O[b,h,n,c] * dO[b,h,n,c] in float32, and dQ_accum := 0.
 * Reads O, dO; writes D and every element of dQ_accum (bf16 with
 * FA_FLAG_DETERMINISTIC: dQ_accum is left alone, since fa_bwd overwrites
 * every slice element fa_convert_dq reads). */
fa_status fa_bwd_preprocess(const fa_problem* p, const void* O, const void* dO,
                            float* D, float* dQ_accum, void* stream);

/* Main backward (ch.16 §16.2, §16.3, §16.6): for each key block K_j, V_j,
 * for each query block Q_i that the causal mask leaves partly visible:
 *   S = scale Q_i K_j^T, P = exp(S - L_i) (masked entries 0),
 *   dV_j += P^T dO_i,  dP = dO_i V_j^T,  dS = P * (dP - D_i),
 *   dQ_accum[i] += dS K_j  (float32 reductions the kernel does not wait
 *                           for; no scale),
 *   dK_j += dS^T Q_i.
 * Writes dV_j and scale * dK_j once per key block.  dQ_accum must hold the
 * zeros written by fa_bwd_preprocess (or earlier partial sums to add to). */
fa_status fa_bwd(const fa_problem* p, const void* Q, const void* K, const void* V,
                 const void* dO, const float* L, const float* D, float* dQ_accum,
                 void* dK, void* dV, void* stream);

/* fa_bwd with tile-pair accounting, to check the causal skip on the device
 * (CS349E lecture 11 demo 4: a causal backward over T x T square blocks needs
 * only the T(T+1)/2 pairs that hold a visible entry, a fraction 1/2 + 1/(2T);
 * ch.16 §16.8 item 2: fully masked tiles are neither loaded nor computed).
 * Same arguments and results as fa_bwd, plus:
 *   counts      device array of two unsigned 64-bit words, 8-byte aligned,
 *               owned and zeroed by the caller; the kernel adds the number of
 *               (key block, query block) pairs it executed to counts[0] and
 *               the number of those with no visible entry to counts[1]
 *   key_rows, query_rows   host int32, set before the launch to the block
 *               heights of the kernel that runs: 128 x 128 for bf16 with
 *               d <= 128; 128 keys x 64 queries at d = 256 (the two
 *               column-half CTAs of a key block execute each pair, which is
 *               counted once); 64 x 64 for fp32 (32 x 32 at d = 256).
 * The counting costs one register update per pair in the MMA-issuing warp;
 * fa_bwd runs the same kernels with counting off. */
fa_status fa_bwd_tile_pair_count(const fa_problem* p, const void* Q, const void* K, const void* V,
                                 const void* dO, const float* L, const float* D, float* dQ_accum,
                                 void* dK, void* dV, unsigned long long* counts, int32_t* key_rows,
                                 int32_t* query_rows, void* stream);

/* dQ = dtype(scale * dQ_accum) (ch.16 §16.3: the convert kernel applies the
 * softmax scale and casts; with FA_FLAG_DETERMINISTIC it first sums the key
 * blocks' slices in increasing order).  Reads dQ_accum, writes dQ.  When dQ
 * and its byte strides are multiples of 32 bytes the kernel writes each
 * 16-column piece of a row with one 256-bit store, else with 128-bit stores;
 * the values written are the same. */
fa_status fa_convert_dq(const fa_problem* p, const float* dQ_accum, void* dQ, void* stream);

/* The three backward calls in order: preprocess, bwd, convert. */
fa_status fa_backward(const fa_problem* p, const void* Q, const void* K, const void* V,
                      const void* O, const void* dO, const float* L, float* D,
                      float* dQ_accum, void* dQ, void* dK, void* dV, void* stream);

/* The same backward as fa_backward in one kernel launch: the preprocess
 * (ch.16 §16.8 item 1), the main kernel and the convert (§16.3) as items of
 * one grid; the pages launch them separately.  Each CTA of the grid takes a
 * ticket in the order CTAs
 * start and the ticket names its item: one query tile's D and zeroed
 * accumulator tile, one key block of the backward, or one query tile's
 * conversion.  Items only wait (bounded) for items with smaller tickets, so
 * the preprocess of the next group of heads and the conversion of the
 * previous one overlap the backward of the current one.  Only bf16 problems
 * with d <= 128; others return FA_ERR_UNSUPPORTED.  D and dQ_accum as for fa_backward; sync: device
 * int32 array of fa_backward_fused_sync_elems(p) elements, scratch owned by
 * the caller (zeroed on `stream` before the launch).  Same results as
 * fa_backward (bitwise with FA_FLAG_DETERMINISTIC). */
size_t fa_backward_fused_sync_elems(const fa_problem* p);
fa_status fa_backward_fused(const fa_problem* p, const void* Q, const void* K, const void* V,
                            const void* O, const void* dO, const float* L, float* D,
                            float* dQ_accum, int32_t* sync, void* dQ, void* dK, void* dV,
                            void* stream);

/* Backward pass for tensors in host memory (page-locked for overlap):
 * Q, O, dO, dQ dense [B, H, N, d] and K, V, dK, dV dense [B, H, N_k, d] host
 * arrays (p's strides must say so: stride_n = d, stride_h = rows*d,
 * stride_b = H*rows*d), L a dense [B, H, N] float32 host array.
 * Heads are independent, so the batch streams through `workspace` (device
 * memory, 256-byte aligned, at least fa_backward_host_workspace_bytes()) in
 * groups of `heads_per_group` heads (0: about eight groups): group c+1 is
 * copied in and group c-1 copied out while group c runs fa_backward on
 * `stream`.  Returns after enqueueing; `stream` continues only once the last
 * result has reached host memory.  Copies use two library-owned streams
 * created on first use per device; concurrent calls on one device (from
 * several host threads) take a per-device lock and enqueue one after the
 * other, so each gets its own results.  No counterpart on the pages: it feeds
 * the backward from host-resident activations. */
size_t fa_backward_host_workspace_bytes(const fa_problem* p, int32_t heads_per_group);
fa_status fa_backward_host(const fa_problem* p, const void* Q, const void* K, const void* V, const void* O,
                           const void* dO, const float* L, void* dQ, void* dK, void* dV, void* workspace,
                           size_t workspace_bytes, int32_t heads_per_group, void* stream);

/* fa_backward without caller-supplied scratch, for callers that cannot
 * allocate device memory (a host framework or plugin that owns all device
 * memory and forbids allocation while it runs, a process with a device-memory
 * budget fixed at start-up, or a loop that cannot afford cudaMalloc's implicit
 * synchronisation).  The paper has no counterpart; this is a deployment
 * convenience.  D and the dQ accumulator live in fixed arrays inside the
 * library (64 MiB accumulator, 4 MiB D; every GPU that loads the library
 * holds them until exit).  Problems with fa_dq_accum_elems(p) > 16 Mi floats
 * or B*H*N > 1 Mi rows return FA_ERR_UNSUPPORTED.  The first call on a device
 * looks up the arrays' device addresses (make it before any stream capture).
 * All calls share the arrays: calls that overlap on the GPU race, so order
 * them on one stream.  Allocates nothing. */
fa_status fa_backward_static_workspace(const fa_problem* p, const void* Q, const void* K, const void* V,
                                       const void* O, const void* dO, const float* L, void* dQ, void* dK,
                                       void* dV, void* stream);

/* Synchronises `stream`, then reads and clears the current device's status
 * word.  *code receives FA_OK or the first device-side error recorded since
 * the last read.  Returns FA_ERR_CUDA if the synchronisation fails. */
fa_status fa_get_device_status(void* stream, int32_t* code);

/* Upper bound, in nanoseconds, of every wait inside the tensor-core kernels
 * (default 2e9).  After it runs out a kernel records FA_ERR_TIMEOUT, drains
 * its own copies in flight, frees its tensor memory and returns. */
void fa_set_wait_limit_ns(uint64_t ns);

/* Failure-detection self test: launches one block that waits on an
 * mbarrier no thread ever arrives at, with the same bounded wait the
 * tensor-core kernels use and a limit of `limit_ns`.  The device status word
 * then holds FA_ERR_TIMEOUT. */
fa_status fa_selftest_wait_timeout(uint64_t limit_ns, void* stream);

const char* fa_status_string(fa_status s);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int32_t fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
