/*
 * ott.h -- C ABI of libott: Outlier Tokens Tracing (OTT) KV-cache
 * quantization on one GB300 (sm_103a): the every-G flush that packs tokens
 * into 2-bit blocks, and the decode-step attention over the three stores.
 *
 * The method: "Accurate KV Cache Quantization with Outlier Tokens Tracing".
 *   zijie-tian.site, sec. 3.1 -- every G tokens the latest group is
 *       quantized to 2 bits; candidates are scored by the key norm.
 *   zijie-tian.site, sec. 3.2 -- an outlier pool of capacity P keeps
 *       full-precision K/V; new tokens compete with pool tokens and a
 *       displaced token is written back to the quantized cache.
 *   zijie-tian.site, sec. 3.3 and flowchart -- decoding multiplies the query
 *       by quantized, residual-window (latest R tokens, fp16) and outlier
 *       keys, softmaxes the concatenated scores and sums the matching values.
 *   sciencestack.ai (arXiv 2505.10938), TL;DR and Abstract -- three KV
 *       caches; keys quantized per channel, values per token; Fig. 1(c) --
 *       keep the tokens whose keys have the smallest magnitude; Fig. 2 --
 *       the decoding and quantization stages.
 *
 * Exact rules this library implements (and the CPU oracle in the test suite
 * implements independently):
 *   - A flush runs when G+R tokens wait unquantized; it takes the G oldest.
 *   - Outlier score: squared L2 norm of the fp16 key, fp32, summed in channel
 *     order. Candidates = pool + group; the P smallest (norm, token index)
 *     stay in the pool (ties to the lower index); all others form the new
 *     block in ascending token order (a block is made at every flush).
 *   - Keys: one fp16 (scale, zero) per channel over the block's tokens.
 *     Values: one fp16 (scale, zero) per token per 32 channels.
 *     mn/mx in fp32 (-0 below +0); s = fp16_rn((mx-mn)/3); z = mn;
 *     code = 0 if s == 0, else clamp(rint((x-z)/s), 0, 3), IEEE fp32 ops.
 *   - Decode attends to every token seen, scale 1/sqrt(d); query head h
 *     reads kv head h / (Hq/Hkv). Output fp16 (round to nearest).
 *
 * Variants, each declared below with its own rules: batches whose sequences
 * differ in length (ott_create_ragged), a paged block pool with sequences
 * that finish and are replaced (ott_create_paged, ott_release_seq,
 * ott_prefill_seq), the cold-pool eviction policy (ott_create_cold), the
 * channel-conditioned outlier criterion (ott_create_pct), Top-K sparse
 * decode (ott_decode_attn_topk), an allocation-free decode
 * (ott_decode_attn_static), and whole steps fed from pinned host memory
 * (ott_step_host). Two diagnostics support measurements (ott_hbm_copy,
 * ott_ex2_probe).
 *
 * Kernels of consecutive calls on one stream are chained by programmatic
 * dependent launches: an append or a decode may start while the kernel
 * before it finishes, and waits for it before reading its inputs.
 *
 * Conventions for every call:
 *   - Device pointers are CUDA device addresses of fp16 data (IEEE binary16),
 *     contiguous, 16-byte aligned. The caller owns them and keeps them alive
 *     until the work queued on `stream` completes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy stream). All
 *     work is queued on it; no call synchronizes except the create and
 *     destroy calls, ott_export_state, ott_export_cold and ott_check_device.
 *   - Arguments and state are checked before anything is queued: a call that
 *     returns an error other than OTT_ERR_CUDA leaves the cache unchanged.
 *     A CUDA error poisons the handle: later calls return OTT_ERR_STATE.
 *   - A handle is not thread-safe. Distinct handles are independent.
 *   - Every sequence of the batch has the same length T, except in the
 *     ragged and paged variants.
 */
#ifndef OTT_H
#define OTT_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ott_cache ott_cache;

enum {
    OTT_OK = 0,
    OTT_ERR_INVALID = -1,   /* bad argument: NULL, misaligned, unsupported shape */
    OTT_ERR_STATE = -2,     /* not allowed now: prefill on a non-empty cache,
                               decode on an empty one, poisoned handle */
    OTT_ERR_CAPACITY = -3,  /* would exceed max_tokens */
    OTT_ERR_OOM = -4,       /* device allocation failed in ott_create */
    OTT_ERR_CUDA = -5,      /* a CUDA call or kernel failed; handle poisoned */
    OTT_ERR_DEVICE = -6     /* a kernel reported a bounded wait that timed out */
};

/*
 * Create an empty cache for B sequences, Hq query heads, Hkv kv heads, head
 * dim d, group G, residual window R, pool capacity P (the pages' defaults are
 * G=128, R=32, P=32). max_tokens bounds T; all device memory is allocated
 * here (blocks, residual ring, pool, split-K scratch). The other calls
 * allocate nothing, except ott_export_state's staging buffer and the
 * parallel prefill's stream-ordered scratch (see ott_prefill).
 * Supported: d in {64, 128}; Hq % Hkv == 0 (any ratio g = Hq/Hkv); G >= 1;
 * R >= 0; P >= 0; (P + G) * (d + 8) * 4 bytes of flush staging must fit in
 * one CTA's shared memory. Uses the current CUDA device.
 * The decode serves up to 4 query heads of a kv head per read of its blocks:
 * g in {1, 2, 4} reads each block once per call, any other g reads it
 * ceil(g / 4) times (the kv head's query heads in slices of 4, the last
 * slice padded with copies of its last head, whose results are dropped).
 * Returns OTT_OK and *out, or an error with *out = NULL.
 */
int ott_create(int B, int Hq, int Hkv, int d, int G, int R, int P,
               int max_tokens, ott_cache **out);

/*
 * As ott_create, for a batch whose sequences may differ in length: the pages
 * state the method for one sequence, and a serving batch holds sequences of
 * different lengths, each quantized, pooled and flushed on its own schedule
 * (zijie-tian.site sec. 3.1 and 3.2 applied per sequence). Additionally
 * requires B <= 256. The split-K scratch is sized for ranges of work that
 * cross many short sequences, so it is larger than ott_create's. Such a
 * cache accepts ott_prefill (all sequences equally long) or
 * ott_prefill_lens (one length per sequence).
 */
int ott_create_ragged(int B, int Hq, int Hkv, int d, int G, int R, int P,
                      int max_tokens, ott_cache **out);

/*
 * As ott_create, with the cold-pool eviction policy of zijie-tian.site
 * sec. 3.2 (the alternative to writing a displaced token back to the main
 * cache; the page sizes the cold pool at 32 tokens). At a flush the pool
 * tokens displaced by the group do not join the new block: they enter the
 * unit's cold pool, C fp16 slots used first in, first out, in ascending token
 * order; once it holds C tokens each new one discards the one that entered
 * first, which no store holds afterwards. The new block is the group's tokens
 * that did not enter the pool, so block sizes depend on the data (see
 * ott_export_cold). ott_decode_attn attends the cold pool like the outlier
 * pool. 0 <= C <= OTT_COLD_MAX; C = 0 discards displaced tokens at once.
 * All sequences have one length (no ott_prefill_lens).
 */
#define OTT_COLD_MAX 4096
int ott_create_cold(int B, int Hq, int Hkv, int d, int G, int R, int P, int C,
                    int max_tokens, ott_cache **out);

/*
 * As ott_create, with the channel-conditioned outlier criterion of
 * zijie-tian.site sec. 3.1 (an outlier token lies in an outlier channel and
 * its magnitude is among the globally smallest p%) in place of the norm
 * ranking. At each flush, over the candidates (the pool plus the group):
 * the outlier channels are the n_oc channels with the largest max |k| (ties
 * to the lower channel index); each candidate's score is its squared key
 * norm over those channels only (fp32, ascending channel order; old pool
 * tokens are scored again, since the channels change from flush to flush);
 * the m = ceil(pct * candidates / 10000) smallest scores (ties to the lower
 * token index) are the outliers, and the pool keeps the min(P, m) most
 * outlying of them. Every other candidate joins the new block (written
 * back). Pool and block sizes follow from (P, G, pct) alone, the same for
 * every unit: pool_j = min(P, ceil(pct * (pool_{j-1} + G) / 10000)), as
 * ott_get_counts and ott_block_count report. pct = 10000 with n_oc = d is the
 * norm criterion of ott_create; pct = 0 keeps no pool. 0 <= pct <= 10000,
 * 1 <= n_oc <= d, else OTT_ERR_INVALID. All sequences have one length.
 */
int ott_create_pct(int B, int Hq, int Hkv, int d, int G, int R, int P, int pct, int n_oc,
                   int max_tokens, ott_cache **out);

/*
 * As ott_create_ragged, with the quantized blocks of all (sequence, kv head)
 * units drawn from one pool of pool_blocks blocks (a paged block table)
 * instead of max_tokens worth of blocks per unit: a serving batch whose
 * sequences differ in length needs only the blocks its tokens fill. Each
 * flush takes one free block per flushed unit; ott_release_seq returns a
 * sequence's blocks. A call whose flushes would need more blocks than are
 * free returns OTT_ERR_CAPACITY before anything is queued. The decode reads
 * every block through the table, so the cache keeps per-sequence counts even
 * after ott_prefill (ott_get_counts then reports sequence 0).
 */
int ott_create_paged(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens,
                     long long pool_blocks, ott_cache **out);

/*
 * Serving (caches from ott_create_ragged or ott_create_paged): sequence b
 * finishes. It drops all its tokens and (paged pool) returns its blocks; the
 * slot must be refilled with ott_prefill_seq before the next ott_append or
 * decode (which return OTT_ERR_STATE while a sequence is empty). Releasing an
 * empty sequence does nothing. With per-sequence counts, max_tokens bounds
 * each sequence: a loop that releases and refills sequences can run for any
 * number of steps as long as no single sequence outgrows max_tokens.
 * stream: the stream of the cache's other calls.
 */
int ott_release_seq(ott_cache *c, int b, void *stream);

/*
 * Serving: fill the empty sequence b with a new prompt of L tokens; from then
 * on it is a fresh sequence of its own (token indices from 0), flushed and
 * attended as in ott_prefill_lens. K, V: DEVICE fp16 [Hkv][L][d], contiguous.
 * An empty cache from ott_create_ragged or ott_create_paged may be filled
 * this way one sequence at a time (appends and decodes wait until every
 * sequence holds a token). OTT_ERR_STATE if b holds tokens; OTT_ERR_CAPACITY
 * if L > max_tokens or the paged pool lacks free blocks.
 */
int ott_prefill_seq(ott_cache *c, int b, const void *K, const void *V, int L, void *stream);

/* Free blocks of a paged pool (host-side count), or -1 for a cache without one. */
long long ott_free_blocks(const ott_cache *c);

/* Free everything. NULL-safe. Waits for the device to finish. */
int ott_destroy(ott_cache *c);

/*
 * Prefill L tokens into an EMPTY cache. K, V: device fp16 [B][Hkv][L][d].
 * Equivalent to L appends in token order (the flush runs for every group of
 * G that leaves the residual window). L may be 0. Errors: OTT_ERR_STATE if
 * T > 0, OTT_ERR_CAPACITY if L > max_tokens.
 * With fewer (sequence, kv head) units than SMs, the flushes run as one
 * parallel pass (the pool after every group found by a scan first), with
 * 16 * P bytes of scratch per (unit, group) allocated on the stream from a
 * pool the library keeps per device (it holds up to 1 GiB between calls);
 * the same applies to ott_prefill_lens and ott_prefill_seq. If no scratch
 * can be had, the flushes run group by group instead.
 */
int ott_prefill(ott_cache *c, const void *K, const void *V, int L, void *stream);

/*
 * Ragged prefill into an EMPTY cache made by ott_create_ragged. K, V: device
 * fp16 [B][Hkv][Lmax][d]; lens: HOST int32[B], read during the call, with
 * 1 <= lens[b] <= Lmax <= max_tokens. Sequence b takes its first lens[b]
 * tokens (the rest of its rows are not read), equivalent to lens[b] appends
 * to that sequence alone. Afterwards every sequence keeps its own token
 * count: ott_append adds one token to each and flushes exactly the
 * sequences whose residual window reached G+R; ott_decode_attn attends each
 * sequence over its own tokens. Errors: OTT_ERR_STATE if the cache is not
 * ragged-capable or not empty, OTT_ERR_INVALID for a length outside
 * [1, Lmax], OTT_ERR_CAPACITY if Lmax > max_tokens.
 */
int ott_prefill_lens(ott_cache *c, const void *K, const void *V, const int *lens, int Lmax,
                     void *stream);

/*
 * Append one token to every sequence. k, v: device fp16 [B][Hkv][d]. The
 * token goes to the fp16 residual ring; when G+R tokens wait, the flush
 * kernel runs on the same stream (the decision is taken on the host from T,
 * without a device round trip).
 */
int ott_append(ott_cache *c, const void *k, const void *v, void *stream);

/*
 * Decode-step attention for one query token per sequence.
 * q: device fp16 [B][Hq][d]; out: device fp16 [B][Hq][d] (may not alias q).
 * out = softmax(q . K^T / sqrt(d)) V over all T tokens: dequantized blocks,
 * residual ring and outlier pool. Requires T >= 1 (else OTT_ERR_STATE).
 * Uses the split-K scratch allocated at create; queues two kernels.
 */
int ott_decode_attn(ott_cache *c, const void *q, void *out, void *stream);

/*
 * One decode step fed from and answered into pinned host memory: the same
 * work as copying k, v and q to the device, ott_append(k, v) and
 * ott_decode_attn(q, out) (topk >= 1: ott_decode_attn_topk(q, out, topk)),
 * then copying out back, but the kernels read and
 * write the host buffers themselves through the device's mapping of pinned
 * memory, so the step is one chain of kernels on the stream with no copy
 * between them (each kernel's launch then overlaps the one before it).
 * k, v: fp16 [B][Hkv][d], q: fp16 [B][Hq][d], out: fp16 [B][Hq][d], all in
 * pinned (page-locked, mapped) host memory, 16-byte aligned; out may not
 * alias an input. The queries are copied to the device by the append kernel.
 * The buffers must stay valid, and the inputs unchanged, until the stream
 * passes the step; out is complete then. A pointer the device cannot address
 * (cudaHostGetDevicePointer fails) or that is not 16-byte aligned gives
 * OTT_ERR_INVALID before anything is queued; the other errors are those of
 * ott_append and ott_decode_attn. (Where the GPU addresses all host memory,
 * pageable buffers are accepted too, at lower speed.)
 */
int ott_step_host(ott_cache *c, const void *k, const void *v, const void *q, void *out, int topk, void *stream);

/*
 * The same decode as ott_decode_attn, but allocation-free: it calls no
 * cudaMalloc, cudaFree or allocating library routine, and it does not use the
 * split-K scratch that ott_create set aside. Its partial results go to a fixed
 * 32 MiB array in libott's device global memory, which every GPU that loads
 * the library holds until the process exits. It serves callers that may not
 * allocate device memory on their decode path: engines that hand all free
 * memory to their own pool at start-up and allow no later growth, and
 * latency-critical loops that cannot afford the implicit synchronization of
 * an allocation. The paper has no counterpart; this is a deployment variant.
 *   - The first call on a device looks up the array's device address (with
 *     the cache's device current); make that first call before any stream
 *     capture. After a device reset (a new context) the next call looks it
 *     up again; caches created before the reset are gone with it.
 *   - Every call shares the array. Calls that overlap on the GPU (other
 *     streams, other handles) race on it; order them (same stream or events).
 *     Nothing in it needs clearing between calls.
 * Errors: as ott_decode_attn, plus OTT_ERR_STATE if the cache's device is not
 * the current device, and OTT_ERR_CAPACITY if this shape's partials
 * (SMs x 16 warps x (units/warps + 2) x 2 x gs x (d+2) floats, where
 * gs = g for g in {1, 2, 4}, else 4, and units = B x Hkv x ceil(g / gs))
 * exceed the array.
 */
int ott_decode_attn_static(ott_cache *c, const void *q, void *out, void *stream);

/*
 * Top-K sparse decode (zijie-tian.site sec. 6: OTT combined with sparse access
 * to the quantized KV). As ott_decode_attn, but each (sequence, kv head)
 * attends only K of its quantized blocks, next to all its residual and pool
 * tokens (and cold-pool tokens under that policy): the non-empty blocks with
 * the largest score bound, ties to the lower block index. The bound of a
 * block for query head h is the largest q.k that a key dequantized from the
 * block's per-channel scale s and zero z can reach, sum over channels of
 * max(q*z, q*(z + 3*s)), in fp32 (round-to-nearest products and sums, channel
 * order); the block's bound is the largest over the query heads that share
 * the kv head. A selected block is attended whole. The bound reads only each
 * block's 4d-byte scale/zero header, so with K well below the block count
 * the call reads far fewer bytes than ott_decode_attn.
 * K >= 1 (K >= the block count attends every block). sel: NULL, or a DEVICE
 * int32 [B*Hkv][min(K, nf)] (nf: the largest block count of any sequence)
 * that receives the selected block indices of each unit in ascending order
 * (-1 where a unit has fewer non-empty blocks), written on the stream. Works
 * on ragged and paged batches: each unit selects among its own blocks.
 * OTT_ERR_INVALID also if the selection's shared memory (about 8 bytes per
 * block slot) does not fit for this max_tokens.
 */
int ott_decode_attn_topk(ott_cache *c, const void *q, void *out, int K, int32_t *sel, void *stream);

/* Counts (same for every sequence and kv head): tokens seen, blocks (flushes),
 * residual tokens, pool tokens. Host-side, no device access. After
 * ott_prefill_lens the counts differ per sequence; this then reports
 * sequence 0 (see ott_get_seq_counts). */
int ott_get_counts(const ott_cache *c, long long *T, int *nf, int *tail, int *n_pool);

/* The same counts for sequence b (0 <= b < B), in either kind of batch. */
int ott_get_seq_counts(const ott_cache *c, int b, long long *T, int *nf, int *tail, int *n_pool);

/* Valid tokens of block j (0 <= j < nf). Host-side. Returns the count or
 * OTT_ERR_INVALID; OTT_ERR_STATE for a cache with the cold-pool policy, whose
 * block sizes differ per unit (ott_export_cold reports them). */
int ott_block_count(const ott_cache *c, int j);

/*
 * Canonical host copy of the state of units [u0, u0+nu), unit = b*Hkv + hkv.
 * Every pointer is a HOST pointer and may be NULL (that array is skipped).
 * Shapes, with nf blocks and nt residual tokens:
 *   bidx  [nu][nf][G]      int32  token indices ascending, -1 padded
 *   kcode [nu][nf][G][d/4] uint8  code of channel c at bits 2(c%4) of byte c/4
 *   ks,kz [nu][nf][d]      fp16 bits: per-channel key scale / zero
 *   vcode [nu][nf][G][d/4] uint8  same packing
 *   vs,vz [nu][nf][G][d/32] fp16 bits: per-token value scale / zero
 *   tk,tv [nu][nt][d]      fp16 bits: residual tokens nf*G .. T-1 in order
 *   pidx  [nu][P] int32 ascending (-1 pad); pnorm [nu][P] fp32 bits;
 *   pk,pv [nu][P][d]       pool tokens in ascending token order (0 padded)
 * Padding slots are zero. Synchronizes the device; allocates a temporary
 * device staging buffer. After ott_prefill_lens the units of one call must
 * belong to one sequence (nf and nt are that sequence's). Errors:
 * OTT_ERR_INVALID for a bad unit range.
 */
typedef struct {
    int32_t *bidx;
    uint8_t *kcode;
    uint16_t *ks, *kz;
    uint8_t *vcode;
    uint16_t *vs, *vz;
    uint16_t *tk, *tv;
    int32_t *pidx;
    uint32_t *pnorm;
    uint16_t *pk, *pv;
} ott_state_export;

int ott_export_state(ott_cache *c, int u0, int nu, const ott_state_export *dst);

/*
 * The cold-pool policy's extra state for units [u0, u0+nu), as HOST arrays
 * (any pointer may be NULL):
 *   bcount [nu][nf] int32   valid tokens of each block (as the decode reads them)
 *   ncold  [nu]     int32   tokens in the cold pool
 *   cidx   [nu][C]  int32   their token indices, the oldest entry first (-1 pad)
 *   ck, cv [nu][C][d]       their fp16 keys and values, same order (0 pad)
 * Synchronizes the device. OTT_ERR_STATE for a cache without the policy.
 */
int ott_export_cold(ott_cache *c, int u0, int nu, int32_t *bcount, int32_t *ncold, int32_t *cidx,
                    uint16_t *ck, uint16_t *cv);

/*
 * Wait for the device and read the cache's device status word: OTT_OK, or
 * OTT_ERR_DEVICE if a kernel gave up a bounded wait, or OTT_ERR_CUDA. After
 * OTT_ERR_DEVICE the handle is poisoned (later calls return OTT_ERR_STATE):
 * the kernel that gave up left its part of the state or the output unwritten.
 */
int ott_check_device(ott_cache *c);

/* Bytes of device memory the cache holds. Host-side. */
long long ott_device_bytes(const ott_cache *c);

/* Static text for a status code. */
const char *ott_status_str(int code);

/*
 * Measurement helper (not part of the method): copy `bytes` from src to dst,
 * both DEVICE pointers, 16-byte aligned, bytes a multiple of 16, ranges not
 * overlapping, with a plain streaming copy kernel on `stream`. A caller times
 * it to measure the HBM bandwidth this GPU sustains (read + write bytes over
 * the elapsed time), the denominator of the decode kernel's roofline
 * fraction, in the same process as the decode timing. Errors:
 * OTT_ERR_INVALID for a bad argument, OTT_ERR_CUDA if the launch fails.
 */
int ott_hbm_copy(void *dst, const void *src, long long bytes, void *stream);

/*
 * Diagnostic (not part of the method): y[i] = 2^x[i] for n DEVICE floats,
 * computed with the same device exponential the decode kernel uses for its
 * softmax weights (the hardware approximation, subnormal results flushed to
 * zero), so that its error against an exact 2^x can be measured. Errors:
 * OTT_ERR_INVALID for a NULL pointer or n < 0, OTT_ERR_CUDA if the launch
 * fails.
 */
int ott_ex2_probe(const float *x, float *y, int n, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OTT_H */
