/*
 * ar.h — C ABI of the GB300 gradient allreduce library (libar.so).
 *
 * N "virtual ranks" live in one GPU's memory: rank r owns an input and an
 * output buffer, and a collective combines all ranks' buffers element by
 * element so that every rank ends with the same result.
 *
 * Sources (web pages on AllReduce), cited by title and section:
 *   [GL] "AllReduce（オールリデュース）" — jisaku.com glossary
 *   [VL] "All-Reduce・All-Gather・All-to-Allとは？LLM分散推論のGPU通信を整理する" — vasteelab
 *   [AW] "AllReduce" — astro-wiki
 *   [WP] "All-reduce" — wikiprompt
 *
 * Conventions for every entry point
 * ---------------------------------
 * Memory and ownership: the caller owns every device buffer, the FP8
 *   workspace and the stream; the library allocates no memory and never
 *   synchronises. Pointer arrays (`sendbufs`, `recvbufs`, `tensors`) and the
 *   count/offset arrays are HOST memory, read during the call only; the
 *   buffers they point to are DEVICE memory of the current device (the
 *   device selected in the calling thread), and `stream` must belong to it
 *   (0 = the legacy default stream).
 * Asynchrony: work is enqueued on `stream` and the call returns at once
 *   (stream separation, [GL] §パフォーマンスチューニング; [VL] §communicationと
 *   computeを重ねる条件). Results are valid after the stream reaches them.
 * Errors: argument errors are detected before anything is enqueued and
 *   return synchronously: AR_ERR_INVALID_ARGUMENT (null pointer, nranks
 *   outside 1..AR_MAX_RANKS, unknown enum, a buffer not aligned to its
 *   element size, workspace too small), AR_ERR_UNSUPPORTED (TREE with a
 *   nranks that is not a power of two; MIN/MAX on the FP8 path; FP8 output
 *   type I32), AR_ERR_ALIAS (buffers overlap other than in the documented
 *   in-place forms). A failed launch returns AR_ERR_CUDA; ar_last_error()
 *   holds the CUDA message. Faults inside kernels surface at the caller's
 *   next synchronisation, as with any CUDA work. On any error nothing has
 *   been written.
 * Counts: `count == 0` (or an empty tensor list) is a successful no-op.
 * Alignment: any element-aligned address works. When every pointer and the
 *   chunk length allow 16-byte vectors the kernels use them; otherwise they
 *   fall back to element-wide accesses with bit-identical results.
 * Numerics: bf16/fp16 inputs widen exactly to binary32, reduce in binary32,
 *   and round once to the output type (nearest even). int32 sums wrap modulo
 *   2^32; int32 AVG truncates toward zero. AVG divides the finished sum once
 *   by nranks (IEEE division for floats). MIN/MAX order -0 below +0 and turn
 *   any NaN input into the canonical quiet NaN of the type (f32 0x7FC00000,
 *   bf16 0x7FC0, fp16 0x7E00). SUM/AVG with NaN inputs return a NaN of
 *   unspecified payload.
 */
#ifndef AR_GB300_H
#define AR_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the runtime's cudaStream_t). */
typedef struct CUstream_st *ar_stream_t;

typedef enum {
    AR_SUCCESS = 0,
    AR_ERR_INVALID_ARGUMENT = 1,
    AR_ERR_UNSUPPORTED = 2,
    AR_ERR_ALIAS = 3,
    AR_ERR_CUDA = 4,
    AR_ERR_TIMEOUT = 5,
    AR_ERR_MISMATCH = 6
} ar_status_t;

typedef enum { AR_F32 = 0, AR_F16 = 1, AR_BF16 = 2, AR_I32 = 3 } ar_dtype_t;

/* Element-wise operators named in [WP] §definition (sum, min, max, average). */
typedef enum { AR_SUM = 0, AR_AVG = 1, AR_MIN = 2, AR_MAX = 3 } ar_op_t;

/* Summation orders / kernel shapes:
 *   AR_ALGO_RING  — ring reduce-scatter kernel, then ring all-gather kernel
 *                   ([GL] §Ring-AllReduceの仕組み; [AW] §Ring AllReduce).
 *   AR_ALGO_FUSED — one pass: the same ring order, every element reduced once
 *                   and stored to all N outputs. Bit-identical to RING.
 *   AR_ALGO_TREE  — one pass in recursive-halving order ([GL] algorithm table,
 *                   "Recursive Halving-Doubling"; [AW] §其他 AllReduce 算法):
 *                   v_r = x_r; for d = N/2, ..., 1: v_r = v_r (+) v_{r+d}, r < d.
 * Ring order: the ranks' data are split into N chunks ([GL] §Ring-AllReduce
 * の仕組み, "N個のチャンクに分割"); chunk c covers elements
 * [c*L, min((c+1)*L, count)), L = ceil(count/N) rounded up to a multiple of
 * 16 bytes / element size (trailing chunks may be short or empty). Chunk c is
 * folded starting at rank c+1: x_{c+1}, x_{c+2}, ..., x_{c+N} (mod N), and
 * rank c ends holding it.
 *   AR_ALGO_STEP_RING — the ring executed literally, one launch per step:
 *                   N-1 reduce-scatter steps (every rank adds the partial it
 *                   receives from rank r-1 to its own chunk) and N-1 all-gather
 *                   steps (every rank forwards a finished chunk to r+1).
 *                   Same bits as RING; moves 5(N-1)*M bytes in 2(N-1) launches.
 *   AR_ALGO_STEP_TREE — recursive halving reduce-scatter (partners at
 *                   distance N/2, N/4, ..., 1 exchange halves of their
 *                   segment) then recursive doubling all-gather ([AW] table,
 *                   Rabenseifner). Same bits as TREE; 5(N-1)*M bytes in
 *                   2*log2(N) launches.
 *   Through ar_allreduce the stepwise orders keep partial sums in the output
 *   buffers, so they take 4-byte element types (F32, I32) only
 *   (AR_ERR_UNSUPPORTED otherwise); ar_allreduce_stepwise runs them for
 *   BF16 and F16 with binary32 partials in a caller workspace.
 *   AR_ALGO_AUTO      — chosen by the library: the one-pass FUSED kernel, which
 *                   measured fastest at every message size on one device. */
typedef enum {
    AR_ALGO_RING = 0,
    AR_ALGO_FUSED = 1,
    AR_ALGO_TREE = 2,
    AR_ALGO_STEP_RING = 3,
    AR_ALGO_STEP_TREE = 4,
    AR_ALGO_AUTO = 5
} ar_algo_t;

#define AR_MAX_RANKS 64
#define AR_FP8_BLOCK 128

/* Allreduce ([GL] §AllReduceの基本動作: every process ends with the same
 * reduced tensor; [VL] §All-Reduceは全rankの値を集約して全rankへ返す; [AW]
 * §定义: N processes with equal-length data).
 *   sendbufs[r] — rank r's input: `count` elements of `dtype` (device).
 *   recvbufs[r] — rank r's output: `count` elements (device). After the call
 *                 every recvbufs[r] holds the same bytes.
 * In place: recvbufs[r] == sendbufs[r] is allowed for any r. Otherwise the
 * output buffers must not overlap each other or any input; inputs may
 * overlap each other (they are only read). */
ar_status_t ar_allreduce(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                         ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, ar_stream_t stream);

/* Workspace bytes of ar_allreduce_stepwise for BF16/F16: one binary32
 * partial array of `count` values per rank (each rounded up to 256 bytes);
 * 0 for other types (they need none) or when nranks or count is out of
 * range. */
size_t ar_stepwise_workspace_bytes(int nranks, size_t count, ar_dtype_t dtype);

/* The stepwise orders (AR_ALGO_STEP_RING, AR_ALGO_STEP_TREE; the literal
 * ring and recursive halving-doubling of [GL]'s algorithm table, one launch
 * per step) for every element type. BF16/F16 inputs are widened exactly, the
 * reduce-scatter steps keep their partial sums in binary32 in `workspace`
 * (device, at least ar_stepwise_workspace_bytes, 16-byte aligned, owned by
 * the caller, contents meaningless before and after), and the last step
 * rounds once to the output type, so the results are bit-identical to
 * AR_ALGO_RING / AR_ALGO_TREE; the all-gather steps copy 16-bit values. F32
 * and I32 need no workspace (it may be null) and run as ar_allreduce does.
 * Other algo values give AR_ERR_INVALID_ARGUMENT; the workspace must not
 * overlap any buffer (AR_ERR_ALIAS). In place and other rules: as
 * ar_allreduce. */
ar_status_t ar_allreduce_stepwise(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                                  ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, void *workspace, size_t ws_bytes,
                                  ar_stream_t stream);

/* A slice of an allreduce: elements [first, first + n) of the result of
 * ar_allreduce over `count` elements per rank, bit-identical to them (same
 * chunk plan, same summation order), computed from those elements alone.
 * The pages have no counterpart: this is how several GPUs share one problem,
 * each holding a contiguous slice of every rank's buffer, with no exchange
 * between them (the result of element i depends only on the N values at i).
 *   sendbufs[r], recvbufs[r] — rank r's slice (n elements each, device):
 *                 element j of the slice is element first + j of the problem.
 *   algo        — RING, FUSED, AUTO and STEP_RING give the ring order, TREE
 *                 and STEP_TREE the recursive-halving order; one launch, or
 *                 two in the ring order when the slice starts inside a chunk.
 * In place and overlap rules: as ar_allreduce. first + n > count gives
 * AR_ERR_INVALID_ARGUMENT; n == 0 is a no-op. */
ar_status_t ar_allreduce_slice(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                               size_t first, size_t n, ar_dtype_t dtype, ar_op_t op, ar_algo_t algo,
                               ar_stream_t stream);

/* Reduce-scatter ([VL] §Reduce-Scatterは集約後の結果をrankへ分ける: reduce
 * element-wise, split into equal chunks, rank r keeps chunk r; [AW]
 * primitives table). Ring order with chunk length `recvcount`.
 *   sendbufs[r] — nranks*recvcount elements (device).
 *   recvbufs[c] — recvcount elements: chunk c of the reduction (device).
 * In place: recvbufs[c] == sendbufs[c] + c*recvcount elements. */
ar_status_t ar_reduce_scatter(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t recvcount,
                              ar_dtype_t dtype, ar_op_t op, ar_stream_t stream);

/* All-gather ([VL] §All-Gatherは分割dataを連結して全rankへ配る: every rank
 * receives all slices concatenated in rank order; [AW] primitives table).
 *   sendbufs[r] — sendcount elements (device).
 *   recvbufs[q] — nranks*sendcount elements; slice r lands at
 *                 recvbufs[q] + r*sendcount for every q (device).
 * In place: sendbufs[r] == recvbufs[r] + r*sendcount elements. A pure copy:
 * dtype only fixes the element size. */
ar_status_t ar_all_gather(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t sendcount,
                          ar_dtype_t dtype, ar_stream_t stream);

/* Bucket plan (host only, no CUDA call). [GL] §パフォーマンスチューニング:
 * several small gradient tensors are packed into one bucket per allreduce,
 * 25 MB by default in PyTorch DDP; [AW] §计算-通信重叠: gradients become ready
 * from the output layer backwards. Tensors are walked in reverse index order;
 * a tensor joins the open bucket if it is empty or if the tensor's end
 * (offset rounded up to 16 bytes, plus its size) stays within cap_bytes;
 * otherwise the bucket closes and a new one starts with it.
 *   counts[t]         — elements of tensor t (host, ntensors entries).
 *   bucket_of[t]      — out: bucket index of tensor t.
 *   offset_of[t]      — out: element offset of tensor t in its bucket
 *                       (a multiple of 16 bytes / element size).
 *   bucket_counts[b]  — out: elements in bucket b (end of its last tensor);
 *                       the caller provides room for ntensors entries.
 *   nbuckets          — out: number of buckets.
 * Padding elements between tensors are not written by flatten. */
ar_status_t ar_bucket_plan(const size_t *counts, int ntensors, ar_dtype_t dtype, size_t cap_bytes,
                           int *bucket_of, size_t *offset_of, size_t *bucket_counts, int *nbuckets);

/* Flatten: bucket[offsets[t] + i] = tensors[t][i] for i < counts[t].
 *   tensors[t] — device pointers (host array of ntensors); offsets in
 *   elements of `dtype` from `bucket` (device). Offsets may address several
 *   ranks' buckets laid out back to back, so one call can flatten every rank.
 * Destination ranges must not overlap each other or any source. */
ar_status_t ar_bucket_flatten(const void *const *tensors, const size_t *counts, const size_t *offsets, int ntensors,
                              ar_dtype_t dtype, void *bucket, ar_stream_t stream);

/* Unflatten: tensors[t][i] = bucket[offsets[t] + i]. Same layout rules. */
ar_status_t ar_bucket_unflatten(const void *bucket, void *const *tensors, const size_t *counts, const size_t *offsets,
                                int ntensors, ar_dtype_t dtype, ar_stream_t stream);

/* Bucket allreduce from the gradient tensors themselves (no flat bucket).
 * Same result, bit for bit, as flattening every rank's tensors into a bucket
 * of bucket_count elements at `offsets`, ar_allreduce on the buckets, and
 * unflattening ([GL] §パフォーマンスチューニング: bucketing; [AW] §计算-通信
 * 重叠: a bucket's allreduce starts as soon as its gradients are ready), but
 * each rank's tensors are read where they live and the result is written to
 * every rank's output tensors directly: 2*N*B bytes moved instead of 6*N*B.
 *   tensors[r*ntensors + t]     — rank r's tensor t (device), counts[t]
 *                                 elements of dtype; host array of
 *                                 nranks*ntensors pointers, rank-major.
 *   out_tensors[r*ntensors + t] — where rank r's reduced tensor t goes; may
 *                                 equal tensors[r*ntensors + t] (in place).
 *   counts, offsets             — host arrays of ntensors entries: element
 *                                 count and element offset of tensor t in the
 *                                 bucket layout (as ar_bucket_plan gives).
 *   bucket_count                — elements in the bucket (fixes the chunks).
 * algo: RING and FUSED give the same bits (the ring order, computed in one
 * pass); TREE is recursive halving (nranks a power of two). Output tensors
 * must not overlap each other or any input other than their own. */
ar_status_t ar_bucket_allreduce(const void *const *tensors, void *const *out_tensors, int nranks, int ntensors,
                                const size_t *counts, const size_t *offsets, size_t bucket_count, ar_dtype_t dtype,
                                ar_op_t op, ar_algo_t algo, ar_stream_t stream);

/* FP8 gradient compression ([GL] §NCCLにおけるAllReduce: FP8 AllReduce halves
 * the traffic; §勾配圧縮技術: FP8 quantisation; [VL] §data typeと圧縮は品質だけ
 * の問題ではない: quantise, dequantise and a scale exchange are needed and the
 * aggregation precision must be managed). Each rank's flat buffer is cut
 * into blocks of AR_FP8_BLOCK = 128 consecutive elements (the last block may
 * be shorter); per block amax = max|x| in binary32, s = amax / 448, and
 * q = E4M3(x / s) rounded to nearest even with saturation to +-448
 * (amax == 0 gives s = 0 and q = 0). The maximum propagates a NaN, so a
 * block holding a NaN has s = NaN and dequantises to NaN throughout, on every
 * FP8 entry point; a block holding an infinity has s = inf and dequantises
 * to NaN as well (inf/inf and 0 * inf).
 *
 * Workspace layout (bytes, all regions 256-byte aligned):
 *   [0, N*QS)            q of rank r at r*QS,  QS = round_up(count, 256)
 *   [N*QS, N*QS + N*SS)  scales of rank r at N*QS + r*SS,
 *                        SS = round_up(ceil(count/128), 64) * 4 */
size_t ar_fp8_workspace_bytes(int nranks, size_t count);

/* Quantise one buffer: in (count elements of in_dtype, F32/F16/BF16) ->
 * q (count bytes, E4M3) and scales (ceil(count/128) floats). Device memory. */
ar_status_t ar_quantize_fp8_blocks(const void *in, ar_dtype_t in_dtype, size_t count, uint8_t *q, float *scales,
                                   ar_stream_t stream);

/* FP8-compressed allreduce: every rank is quantised once into `workspace`
 * (the wire format), then the dequantised values float(q)*s (one binary32
 * multiply) are reduced in binary32 in the order `algo` names, SUM or AVG,
 * rounded once to out_dtype (F32/F16/BF16) and written to every recvbufs[r].
 * RING = reduce-scatter into each owner's chunk, then all-gather copies;
 * FUSED = one pass writing all N outputs; TREE = recursive halving.
 * Chunks use 16 bytes / out_dtype size. recvbufs must not overlap sendbufs
 * or the workspace; ws_bytes >= ar_fp8_workspace_bytes(nranks, count). */
ar_status_t ar_allreduce_fp8(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                             ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_algo_t algo,
                             void *workspace, size_t ws_bytes, ar_stream_t stream);

/* FP8-compressed allreduce with the quantisation fused into the reduction:
 * the same bits as ar_allreduce_fp8 with the same arguments (every rank's
 * blocks quantised once, dequantised, reduced in binary32 in the order `algo`
 * names), but the E4M3 codes and scales stay in registers instead of a wire
 * buffer, so no workspace is needed and the call moves 2*N*M bytes instead
 * of 2*N*M + 2*N*(M/2 + M/64). ([GL] §勾配圧縮技術: FP8 quantisation;
 * [VL] §data typeと圧縮: quantise/dequantise and scale handling cost extra
 * kernels and bytes — here they are folded into the one pass.)
 * RING and FUSED give the same bits; TREE is recursive halving. 16-bit
 * inputs need a 16-bit output type (AR_ERR_UNSUPPORTED otherwise).
 * recvbufs must not overlap sendbufs or each other. */
ar_status_t ar_allreduce_fp8_fused(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                                   ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_algo_t algo,
                                   ar_stream_t stream);

/* FP8 re-quantised on every ring hop: what a ring that sends FP8 on the wire
 * computes when partial sums travel compressed ([GL] §NCCLにおけるAllReduce;
 * [VL] §data typeと圧縮: reducing partial results at low precision changes the
 * numerical error). Chunk c starts at rank c+1; before each of the N-1
 * reduce-scatter hops the running partial of every 128-element block (blocks
 * counted from the chunk's start) is quantised to E4M3 (s = amax/448, nearest
 * even, saturating) and dequantised, then the next rank's value is added in
 * binary32; the finished chunk (AVG divides by N) is quantised once more for
 * the all-gather and every rank stores the same dequantised values in
 * out_dtype. Ring order only; SUM or AVG; any F32/F16/BF16 in and out types;
 * element-aligned buffers. recvbufs must not overlap sendbufs or each other.
 * Compare ar_allreduce_fp8, which quantises each rank's input once. */
ar_status_t ar_allreduce_fp8_hops(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                                  ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_stream_t stream);

/* Bytes of the FP8 workspace built into the library (16 MiB per device). */
#define AR_FP8_STATIC_WS_BYTES (16u * 1024u * 1024u)

/* FP8-compressed allreduce for callers that cannot allocate device memory.
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot obtain a workspace for ar_allreduce_fp8: code running inside an
 * allocator's or memory pool's own callbacks, on a framework path where
 * allocation is forbidden, or a host program with no access to the CUDA
 * allocation API. It computes exactly what ar_allreduce_fp8 computes (same
 * kernels, same bits) but keeps the quantised codes and scales in a fixed
 * array inside the library, AR_FP8_STATIC_WS_BYTES bytes on every device that
 * loads it, held until the process exits. It calls no cudaMalloc, cudaFree
 * or other allocating routine.
 *   Limit: ar_fp8_workspace_bytes(nranks, count) must not exceed
 *   AR_FP8_STATIC_WS_BYTES (for example 8 ranks x 2,000,000 elements fit);
 *   larger calls return AR_ERR_INVALID_ARGUMENT and ar_last_error() says why.
 *   Set-up: the first call made in a CUDA context (normally the device's
 *   primary context, so once per device) looks up the array's address in
 *   that context (cudaGetSymbolAddress) and caches it with the context's ID;
 *   make that first call before any stream capture. A later call in another
 *   context, for example after cudaDeviceReset, looks the address up again.
 *   Argument errors are reported as by ar_allreduce_fp8 and take precedence
 *   over the size limit; a count whose workspace size overflows is "count
 *   too large".
 *   Sharing: all calls on a device use the same array and leave their data in
 *   it; each call writes every byte it later reads, so nothing needs
 *   clearing, but calls that overlap on the GPU (different streams, or host
 *   threads sharing a device without ordering) race on it and must be
 *   serialised by the caller.
 * Other arguments, rules and errors: as ar_allreduce_fp8. */
ar_status_t ar_allreduce_fp8_noalloc(const void *const *sendbufs, void *const *recvbufs, int nranks, size_t count,
                                     ar_dtype_t in_dtype, ar_dtype_t out_dtype, ar_op_t op, ar_algo_t algo,
                                     ar_stream_t stream);

/* Top-K gradient sparsification with error feedback ([GL] §勾配圧縮技術: only
 * the largest K% of the gradient is communicated and error feedback makes up
 * for what is dropped; [WP] §优化技术: top-k sends the indices as well). The
 * pages fix no formula or tie rule; this library's reading, per rank r:
 *   a = grads[r] + residuals[r]    (binary32 add, round to nearest even)
 *   keep the k entries of largest |a|; among equal |a| the lower index first
 *   idx[r][0..k), val[r][0..k) = the kept (index, a[index]) in ascending
 *                                 index order
 *   residuals[r] = a with the kept entries set to +0
 * so the dense form of (idx, val) plus the new residual equals a exactly.
 * |a| is compared through its bit pattern with the sign cleared (so -0 ties
 * +0, and a NaN ranks above every number); a = g + e of a NaN is the device's
 * one canonical NaN, so all NaNs tie and the lower index comes first.
 *
 * Workspace bytes for ar_topk_compress over nranks x `count` values keeping
 * k per rank (per rank about 3 * count / 4 + 128 * k bytes, at most 4.25
 * bytes per value, plus 8 KiB; a multiple of 256 bytes);
 * 0 if nranks is outside 1..AR_MAX_RANKS, count >= 2^32 or k > count. */
size_t ar_topk_workspace_bytes(int nranks, size_t count, size_t k);

/* Every rank's Top-K step in one call on `stream` (six kernel launches
 * whatever nranks is): reads grads[r][count], updates residuals[r][count] in
 * place and writes idx[r][k] (uint32 indices) and val[r][k].
 *   grads[r], residuals[r]: F32 device buffers, 4-byte aligned (when all are
 *     16-byte aligned the vector path runs; results are identical either way).
 *   workspace: device memory of at least ar_topk_workspace_bytes(nranks,
 *     count, k), 16-byte aligned, owned by the caller; its contents need no
 *     initialisation. A call leaves in it its threshold, which the next
 *     call on the same workspace uses to collect its candidates (the values
 *     at or above 0.5 to 0.99 times it, a margin that widens after a call
 *     whose threshold fell below it and narrows while it holds) during the
 *     pass that forms a = g + e (large
 *     calls, 16-byte aligned buffers): when at least k values are collected
 *     and they fit, the data is read once instead of twice, and when the
 *     threshold's leading 11 bits also hold, that pass narrows the
 *     selection one step further. Results never depend on the workspace's
 *     contents; a stale or garbage threshold only costs the second pass.
 *   Errors: AR_ERR_INVALID_ARGUMENT for k > count, count >= 2^32, a null or
 *   misaligned pointer or a short workspace; AR_ERR_ALIAS if an output
 *   (residual, idx, val, workspace) overlaps another output or an input
 *   (inputs may overlap each other). k == 0 only folds grads into residuals;
 *   count == 0 is a no-op. */
ar_status_t ar_topk_compress(const float *const *grads, float *const *residuals, int nranks, size_t count,
                             size_t k, uint32_t *const *idx, float *const *val, void *workspace, size_t ws_bytes,
                             ar_stream_t stream);

/* Workspace bytes for ar_sparse_allreduce with SUM or AVG: one uint32 per
 * rank and output tile boundary, 4 * nranks * (ceil(count / T) + 1) rounded
 * up to a multiple of 256, where the tile T is 6144 / nranks rounded down to
 * a multiple of 128 and kept within 128..4096 (768 values at 8 ranks, about
 * count / 24 bytes); 0 if nranks is outside 1..AR_MAX_RANKS or
 * count >= 2^32. */
size_t ar_sparse_workspace_bytes(int nranks, size_t count);

/* Allreduce of sparse vectors ([GL] §勾配圧縮技術): rank r contributes the
 * dense vector of length `count` that is zero except at idx[r][j] where it
 * holds val[r][j] (j < nnz[r]); every recvbufs[r] receives the allreduce of
 * those dense vectors, bit-identical to ar_allreduce of F32 buffers holding
 * them (+0 where absent) with the same op and algo.
 *   SUM, AVG: one pass without dense copies — each tile of the output is
 *     densified in shared memory from every rank's pairs and folded in the
 *     order of `algo`; the output buffers are only written. Needs a device
 *     workspace of ar_sparse_workspace_bytes(nranks, count), 16-byte aligned
 *     (contents need no initialisation), and each rank's indices in strictly
 *     ascending order (ar_topk_compress writes them so). Indices out of
 *     order leave the result unspecified; every access stays inside the
 *     buffers.
 *   MIN, MAX: the outputs are zeroed, the pairs scattered into them and the
 *     dense allreduce run in place; `workspace` is not used (may be null)
 *     and any index order works.
 *   idx[r], val[r]: device arrays of nnz[r] entries; indices must be < count
 *     and distinct within a rank. An index >= count is dropped; which of two
 *     equal indices wins is unspecified.
 *   recvbufs[r]: F32 device buffers of `count`, 4-byte aligned, disjoint from
 *     each other, from the workspace and from every idx/val array.
 *   Errors: as ar_allreduce, plus AR_ERR_INVALID_ARGUMENT for nnz[r] > count,
 *   count >= 2^32, or (SUM, AVG) a missing, misaligned or short workspace. */
ar_status_t ar_sparse_allreduce(const uint32_t *const *idx, const float *const *val, const size_t *nnz, int nranks,
                                size_t count, ar_op_t op, ar_algo_t algo, float *const *recvbufs, void *workspace,
                                size_t ws_bytes, ar_stream_t stream);

/* Host-side communicator for virtual ranks driven by host threads
 * ([VL] §rankとcommunicator: every rank calls the matching collective with the
 * same count and type; §hangをtimeoutだけで再起動しない: hangs come from ranks
 * that skip a call, differ in count or type, call in a different order, or
 * failed earlier; record each rank's last collective, sequence number, shape,
 * type, communicator id and earlier error). Each thread calls
 * ar_comm_allreduce with its rank's buffers; the call blocks until every rank
 * of the communicator has entered its call with the same sequence number,
 * and the last arrival enqueues the one ar_allreduce on `stream`.
 *   AR_ERR_MISMATCH — a rank's count, dtype, op, algo or stream differs from
 *                     the first arrival's (also a different call order):
 *                     nothing is launched, every rank of the call gets it.
 *   AR_ERR_TIMEOUT  — not every rank arrived within timeout_ms: nothing is
 *                     launched; waiting ranks return after the timeout.
 * After either error the communicator is poisoned: every later call returns
 * the same status at once (isolate the group and rebuild it). Waits are on
 * the host only; no kernel waits on another rank. Thread-safe; one thread per
 * rank at a time. */
typedef struct ar_comm ar_comm_t;

/* What a rank last did on a communicator. */
typedef struct {
    uint64_t comm_id;        /* process-unique communicator id */
    uint64_t seq;            /* collectives this rank has entered (1-based) */
    int collective;          /* 1 = allreduce */
    size_t count;            /* elements */
    int dtype, op, algo;     /* as passed */
    int status;              /* outcome (ar_status_t) */
    uint64_t arrived_mask;   /* ranks that had arrived for this call */
    uint64_t mismatch_mask;  /* ranks whose arguments differed */
    double arrival_skew_ms;  /* last arrival minus first arrival so far */
} ar_call_record_t;

ar_status_t ar_comm_create(int nranks, int timeout_ms, ar_comm_t **comm);
ar_status_t ar_comm_destroy(ar_comm_t *comm);
ar_status_t ar_comm_allreduce(ar_comm_t *comm, int rank, const void *sendbuf, void *recvbuf, size_t count,
                              ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, ar_stream_t stream);
ar_status_t ar_comm_last_record(ar_comm_t *comm, int rank, ar_call_record_t *out);

/* Static text for a status code. */
const char *ar_status_string(ar_status_t status);

/* Detail of the last error returned to the calling thread (e.g. the CUDA
 * error text); "" if none. Valid until the thread's next library call. */
const char *ar_last_error(void);

/* Library version string. */
const char *ar_version(void);

#ifdef __cplusplus
}
#endif

#endif /* AR_GB300_H */
