// ott_decode.cu -- decode-step attention over the three OTT stores.
//
// "Accurate KV Cache Quantization with Outlier Tokens Tracing":
// zijie-tian.site sec. 3.3 and the flowchart (the query meets quantized,
// residual-window and outlier keys; the scores are concatenated and
// softmaxed; the weights multiply the matching values and are summed);
// sciencestack.ai Fig. 2 (decoding stage).
//
// Split-K (flash-decoding) design for one GB300:
//   * Work items, unit by unit (unit = (sequence, kv head)): first the fp16
//     tokens (residual ring, then pool) in chunks of 32, then the quantized
//     blocks. A persistent grid (one CTA of 16 warps per SM) gives every warp
//     an equal contiguous range of items (stream-K partition): no atomics, no
//     tail, and one partial (m, l, acc[d]) per query head for each (unit,
//     item type) segment a warp touches. k_combine finds a unit's partials
//     arithmetically and merges them with log-sum-exp weights.
//   * Quantized segments: each warp streams its blocks into a private
//     two-stage shared-memory ring with 1-D TMA bulk copies
//     (cp.async.bulk + mbarrier complete_tx), one copy per chunk of up to
//     4 tiles of 16 tokens. Waits are bounded; a timeout sets the status word.
//   * Dequantization is folded into the products: q.k_hat =
//     sum_c (q_c s_c) code_c + sum_c q_c z_c and
//     p.v_hat = sum_t (p_t s_t) code_t + sum_t p_t z_t.
//     A code word becomes an fp16x2 mma.sync operand with one AND (the code
//     is an exact fp16 subnormal, see ott_internal.cuh); the other operand
//     (q*s or p*s) is split into fp16 hi + lo for fp32-grade products.
//     Scores: A = K codes [16 tokens x 16 channels], B = q*s [16 x (head,
//     hi/lo)]. PV: A = V codes [16 channels x 16 tokens], B = p*s [16 tokens
//     x (head, group, hi/lo)]. All query heads of a kv head share the codes.
//   * fp16 segments: one lane per token for the scores, one lane per d/32
//     channels for P.V, fp32 accumulation, online softmax across chunks.
#include <math_constants.h>

#include <type_traits>

#include "ott_internal.cuh"

namespace ott {
namespace {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// The KV stream is read once per call: its bulk copies carry an L2
// evict-first policy, so that it does not push the split-K partials (read by
// the combine right after) and the queries out of L2.
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_copy_only(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(evict_first_policy())
        : "memory");
}

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    expect_tx(bar, bytes);
    bulk_copy_only(dst, src, bytes, bar);
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: gives up after a fixed number of polls instead of hanging.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    for (int it = 0; it < (1 << 22); ++it)
        if (mbar_try(bar, parity)) return true;
    return false;
}

// 2^x with the hardware approximation (relative error ~2^-22); x <= 0 here,
// -inf gives 0 and results below the normal range flush to 0.
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float pow2i(int k) { return __int_as_float((k + 127) << 23); }

// Two codes at position p of a word as an fp16x2 subnormal pair (class of p);
// w10 = w >> 10. p is a compile-time constant once the callers are unrolled.
__device__ __forceinline__ uint32_t ext_rt(uint32_t w, uint32_t w10, int p) {
    return p < 5 ? (w & (0x00030003u << (2 * p))) : (w10 & (0x00030003u << (2 * (p - 5))));
}

__device__ __forceinline__ uint32_t h2bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

struct DecodeArgs {
    const uint8_t *blk;
    long long blk_bytes;
    int NB;
    const __half *rk, *rv;
    int ring;
    const __half *pk, *pv;
    int P;
    const __half *q;
    __half *out;
    float *part;
    int *ctl;
    int Hq, Hkv, G;
    // a kv head's g = Hq/Hkv query heads are served in S passes of GQ heads
    // (slices); work units are (sequence, kv head, slice), u = (b*Hkv + hkv)*S + s
    int g, S;
    int nf, jfull;      // blocks; blocks j >= jfull hold G tokens
    int ring_start;     // first residual token's ring slot
    int ntail, npool;
    int Sf;             // fp16 items per unit (FP16_CHUNK tokens each)
    int Iu;             // work items per unit: Sf + nf * CPB
    int CPB;            // chunks (CHUNK_TILES tiles) per block
    int IPB;            // quantized work items per block: 1 (whole blocks) or CPB (chunks)
    long long W;        // U * Iu
    int NWp;            // warps in the grid
    int MAXU;           // units a warp's range can touch
    int NSM;            // SMs of the device (the combine's CTA count is sized to them)
    float sl2;          // softmax scale 1/sqrt(d) times log2(e)
    int B;              // sequences (the ragged table's length)
    // cold-pool policy: data-dependent block sizes and a fourth, fp16 store
    const int32_t *bcnt;       // [U][NB] valid tokens of each block
    const __half *ck, *cv;     // [U][C][d] cold pool, a ring used first in, first out
    const int *cmeta;          // [U][2]: tokens in the cold pool, slot of the oldest
    int C;
    // Top-K sparse decode: the quantized items of unit u are the blocks
    // sel[u][0..Ksel) (ascending, -1 for none) instead of blocks 0..nf-1
    const int32_t *sel;
    int Ksel;
    // paged pool (ragged caches from ott_create_paged): block j of unit u is
    // pool slot bt[u*NB + j]; null otherwise
    const int32_t *bt;
};

template <int D, int GQ>
struct Cfg {
    static constexpr int NKT = D / 16;             // score k-tiles = PV m-tiles
    static constexpr int NW = D / 32;              // code words per lane per tile
    static constexpr int NG = D / 32;              // value groups of 32 channels
    static constexpr int GPV = 4 / GQ;             // value groups per PV B variant
    static constexpr int NV = (NG + GPV - 1) / GPV;  // PV B variants
    static constexpr int STAGE = stage_bytes(D);
    static constexpr int QHL = GQ * 2 * (D + 8) * 2;   // per-block hi/lo staging bytes
    // stages, barriers, the queries (fp16, as given) and the hi/lo staging
    static constexpr int WARP_SMEM = 2 * STAGE + 16 + GQ * D * 2 + QHL;
    // the fp16 path stages 8 key and 8 value rows of d+8 halves in each of
    // the same two stage buffers
    static_assert(2 * 8 * (D + 8) * 2 <= STAGE, "fp16 sub-tile staging must fit a stage buffer");
};

// Valid tokens of block j of unit u: fixed by (P, G, j) when displaced pool
// tokens are written back, written by the flush under the cold-pool policy.
template <bool CO>
__device__ __forceinline__ int block_cnt(const DecodeArgs &a, int u, int j) {
    if constexpr (CO) return __ldg(a.bcnt + (size_t)u * a.NB + j);
    return j >= a.jfull ? a.G : block_count(a.P, a.G, j);
}

// First item of warp w's range (items are split as evenly as integers allow).
// The quotients are exact either way; 32-bit division is several times
// cheaper than 64-bit and covers every realistic size.
__device__ __forceinline__ long long range_start(long long W, int NWp, long long w) {
    const unsigned long long num = (unsigned long long)w * (unsigned long long)W;
    if (num <= 0xffffffffull) return (long long)((unsigned)num / (unsigned)NWp);
    return (long long)(num / (unsigned long long)NWp);
}

// The warp whose range holds item x.
__device__ __forceinline__ int warp_of(long long W, int NWp, long long x) {
    const unsigned long long num = (unsigned long long)(x + 1) * (unsigned long long)NWp + (unsigned long long)W - 1;
    if (num <= 0xffffffffull) return (int)((unsigned)num / (unsigned)W) - 1;
    return (int)(num / (unsigned long long)W) - 1;
}

// Unit of item x (x < W).
__device__ __forceinline__ int unit_of(long long x, int Iu) {
    if ((unsigned long long)x <= 0xffffffffull) return (int)((unsigned)x / (unsigned)Iu);
    return (int)(x / Iu);
}

__device__ __forceinline__ size_t part_slot(const DecodeArgs &a, int w, int unit_off, int type) {
    return ((size_t)w * a.MAXU + unit_off) * 2 + type;
}

// Per-sequence counts: scalars in DecodeArgs when every sequence has the
// same length, a table (kernel parameter) when the batch is ragged.
struct NoTable {};
template <bool RG>
using TableT = typename std::conditional<RG, SeqTable, NoTable>::type;

struct UnitInfo {
    long long ub;       // the unit's first work item
    int u, ntail, npool, ring_start, Sf, Iu;
};

// The unit holding work item x (x < W), with its counts.
template <bool RG>
__device__ __forceinline__ UnitInfo unit_at(const DecodeArgs &a, const TableT<RG> &st, long long x) {
    UnitInfo r;
    if constexpr (RG) {
        int lo = 0, hi = a.B;   // e[lo].base <= x < e[hi].base
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (st.e[mid].base <= x) lo = mid;
            else hi = mid;
        }
        const SeqEntry &e = st.e[lo];
        const int h = (int)((unsigned)(x - e.base) / (unsigned)e.Iu);
        r.u = lo * a.Hkv * a.S + h;
        r.ub = e.base + (long long)h * e.Iu;
        r.ntail = e.ntail;
        r.npool = e.npool;
        r.ring_start = e.ring_start;
        r.Sf = e.Sf;
        r.Iu = e.Iu;
    } else {
        r.u = unit_of(x, a.Iu);
        r.ub = (long long)r.u * a.Iu;
        r.ntail = a.ntail;
        r.npool = a.npool;
        r.ring_start = a.ring_start;
        r.Sf = a.Sf;
        r.Iu = a.Iu;
    }
    return r;
}

template <int NW>
__device__ __forceinline__ void lds_words(const uint8_t *p, uint32_t (&w)[NW]) {
    if constexpr (NW == 4) {
        const uint4 x = *reinterpret_cast<const uint4 *>(p);
        w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    } else {
        const uint2 x = *reinterpret_cast<const uint2 *>(p);
        w[0] = x.x; w[1] = x.y;
    }
}

// The GQ query heads of work unit u (a kv-head slice); heads of a padded
// last slice repeat the kv head's last query head (their results are unused).
template <int D, int GQ>
__device__ void load_queries(const DecodeArgs &a, int u, float *qsm, int lane) {
    if (a.S == 1 && a.g == GQ) {
        const int b = u / a.Hkv, hkv = u % a.Hkv;
        const __half2 *qp = reinterpret_cast<const __half2 *>(a.q + ((size_t)b * a.Hq + hkv * GQ) * D);
        for (int e = lane; e < GQ * D / 2; e += 32) reinterpret_cast<__half2 *>(qsm)[e] = qp[e];
    } else {
        const int Hv = a.Hkv * a.S, b = u / Hv, hv = u % Hv, hkv = hv / a.S, h0 = (hv % a.S) * GQ;
        const __half2 *qp = reinterpret_cast<const __half2 *>(a.q + ((size_t)b * a.Hq + (size_t)hkv * a.g) * D);
        for (int e = lane; e < GQ * D / 2; e += 32) {
            const int h = min(h0 + e / (D / 2), a.g - 1);
            reinterpret_cast<__half2 *>(qsm)[e] = qp[h * (D / 2) + e % (D / 2)];
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- quantized segment
// Quantized work items [q0, q1) of kv unit u (queries of work unit uq): item q is the block at position
// q / IPB (Top-K: the block listed there in the unit's selection), whole
// (IPB = 1) or its chunk q % IPB (IPB = CPB: chunks of up to CHUNK_TILES
// tiles); the partial goes to part[slot]. Chunks past a short block's tokens
// hold no work and are skipped.
//
// The chunks are walked by two cursors: one issues the bulk copies two
// chunks ahead, the other consumes them. The first chunk of each block the
// segment meets also brings the block's K scale/zero header. A chunk whose
// tiles are all full (the common case: every block after the pool fills holds
// G tokens) runs a body without any masking; the ragged last chunk of a short
// block takes the masked body.
template <int D, int GQ, bool CO, bool TK, bool RG>
__device__ bool quant_segment(const DecodeArgs &a, size_t slot, int u, int uq, int q0, int q1, uint8_t *stg0,
                              uint8_t *stg1, uint64_t *bars, uint32_t &phase, float *qsm, __half *qhl,
                              int lane) {
    using C = Cfg<D, GQ>;
    constexpr int NKT = C::NKT, NW = C::NW, NG = C::NG, GPV = C::GPV, NV = C::NV;
    constexpr int KSZ = ksz_bytes(D), TB = tile_bytes(D);
    constexpr int CT = CHUNK_TILES * TILE;   // token slots per chunk
    const int r = lane >> 2, i = lane & 3;

    // tokens of the block at position j of the segment (0: no block there)
    auto cnt_at = [&](int j) -> int {
        if constexpr (TK) {
            const int bj = __ldg(a.sel + (size_t)u * a.Ksel + j);
            return bj < 0 ? 0 : block_cnt<CO>(a, u, bj);
        }
        return block_cnt<CO>(a, u, j);
    };
    // chunk cursor: block position j, chunk k of that block, the block's tokens
    struct Cursor {
        int j, k, cnt;
    };
    const int CPB = a.CPB, IPB = a.IPB, KPI = CPB / IPB;   // chunks per item
    const int jl = (q1 - 1) / IPB, kl = ((q1 - 1) % IPB + 1) * KPI - 1;   // the segment's last chunk
    auto past = [&](const Cursor &c) { return c.j > jl || (c.j == jl && c.k > kl); };
    // move to the next chunk that holds tokens (or past the segment)
    auto settle = [&](Cursor &c) {
        while (!past(c) && CT * c.k >= c.cnt) {
            ++c.j;
            c.k = 0;
            c.cnt = c.j <= jl ? cnt_at(c.j) : 0;
        }
    };
    auto advance = [&](Cursor &c) {
        if (++c.k >= CPB) {
            ++c.j;
            c.k = 0;
            c.cnt = c.j <= jl ? cnt_at(c.j) : 0;
        }
        settle(c);
    };
    Cursor ic{q0 / IPB, (q0 % IPB) * KPI, 0};
    ic.cnt = cnt_at(ic.j);
    settle(ic);
    // a block's first chunk in this segment brings the block's header
    const int jf = ic.j, kf = ic.k;
    auto hdr = [&](const Cursor &c) { return c.k == 0 || (c.j == jf && c.k == kf); };
    auto issue = [&](const Cursor &c, int st) {
        if (lane == 0) {
            const int vt = (c.cnt + TILE - 1) / TILE;
            const int t0 = c.k * CHUNK_TILES, nt = min(CHUNK_TILES, vt - t0);
            int bj = c.j;
            if constexpr (TK) bj = __ldg(a.sel + (size_t)u * a.Ksel + c.j);
            size_t bslot = (size_t)u * a.NB + bj;
            if constexpr (RG) {
                if (a.bt) bslot = (size_t)__ldg(a.bt + bslot);
            }
            const uint8_t *bsrc = a.blk + bslot * a.blk_bytes;
            uint8_t *dst = st ? stg1 : stg0;
            if (c.k == 0) {
                bulk_load(dst, bsrc, (uint32_t)(KSZ + nt * TB), &bars[st]);
            } else if (hdr(c)) {   // the header, then the chunk's tiles, on one barrier
                expect_tx(&bars[st], (uint32_t)(KSZ + nt * TB));
                bulk_copy_only(dst, bsrc, (uint32_t)KSZ, &bars[st]);
                bulk_copy_only(dst + KSZ, bsrc + KSZ + (size_t)t0 * TB, (uint32_t)(nt * TB), &bars[st]);
            } else {
                bulk_load(dst + KSZ, bsrc + KSZ + (size_t)t0 * TB, (uint32_t)(nt * TB), &bars[st]);
            }
        }
    };
    // start the copies first (blocks are final here: no flush precedes a
    // programmatic launch), then wait for the kernel this grid depends on,
    // and stage the queries while the copies fly
    Cursor cc = ic;
    int st_issue = 0;
    for (int n = 0; n < 2 && !past(ic); ++n) {
        issue(ic, st_issue);
        st_issue ^= 1;
        advance(ic);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    load_queries<D, GQ>(a, uq, qsm, lane);

    // Cooperative per-block constants: lane L handles channel pairs
    // (2L + 64m, 2L + 64m + 1); the channels' class scales stay in registers
    // for the whole segment.
    constexpr int NPAIR = D / 64;
    float clsf[NPAIR];
    {
#pragma unroll
        for (int m = 0; m < NPAIR; ++m) {
            const int ch = 2 * lane + 64 * m;
            // a channel's slot q = o*NKT + kt (o = bit 3, kt = ch / 16) fixes
            // its class; ch and ch + 1 share the slot
            const int q0 = ((ch >> 3) & 1) * NKT + (ch >> 4);
            clsf[m] = pow2i(-2 * cls_of_pos(q0 & 7));
        }
    }

    float acc[NKT][4];
#pragma unroll
    for (int mt = 0; mt < NKT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    // The two lanes that hold the hi and lo piece of one P.V column (lanes l
    // and l ^ 4) share the work of p*s: with an even number of B variants
    // (GQA) each computes half of the variants, with one variant (MHA) half of
    // the four tokens, both pieces, and receives its piece of the other half
    // from its partner. zs[k] sums variant 2k + piece (split variants) or the
    // lane's two tokens of its one variant.
    static_assert(NV == 1 || NV % 2 == 0, "one or an even number of B variants");
    constexpr bool SPLIT = NV % 2 == 0;
    constexpr int NZ = SPLIT ? NV / 2 : NV;
    static_assert(!SPLIT || NV * GPV == NG, "split variants cover every value group");
    float zs[NZ];
#pragma unroll
    for (int v = 0; v < NZ; ++v) zs[v] = 0.0f;
    float2 zs2 = make_float2(0.0f, 0.0f);   // one variant: the lane's two tokens, kept apart until the end
    // running max and sum of the head this lane's score columns hold
    float m_run = -CUDART_INF_F, l_run = 0.0f;
    uint32_t Bk[NKT][2];
    float c1 = 0.0f, c0 = 0.0f;

    // Score-MMA B column of this lane: head (r/2) mod GQ, piece r&1 (hi or
    // lo). With fewer than four heads the heads repeat across the columns, so
    // that every lane's score columns hold a real head: lane i scores head
    // i mod GQ.
    const int hB = (r >> 1) % GQ;
    const bool piece = (r & 1) != 0;
    const int hS = i % GQ;
    // PV B column of this lane: head hV, value-group offset glow, piece
    const int hV = (r >> 1) / GPV, glow = (r >> 1) % GPV;
    const int src0 = 4 * (2 * i) + hV, src1 = 4 * (2 * i + 1) + hV;
    const bool lo_lane = (r & 1) != 0;
    // One B variant (GQ <= 2): lane (r, i) holds the weights of tokens r and
    // r+8 of head i mod GQ; lanes i with odd i / GQ send the second, so that a
    // hi lane gathers tokens 2i, 2i+1 of head hV and a lo lane tokens 2i+8,
    // 2i+9 with two shuffles
    const int srcA = 4 * (2 * i) + hV + (lo_lane ? GQ : 0), srcB = srcA + 4;
    const bool send_second = ((i / GQ) & 1) != 0;

    int st = 0;
    while (!past(cc)) {
        uint8_t *stage = st ? stg1 : stg0;
        if (!mbar_wait(&bars[st], (phase >> st) & 1u)) {
            if (lane == 0) atomicExch(&a.ctl[1], 1);
            // let the other copy in flight land before giving up the buffers
            mbar_wait(&bars[st ^ 1], (phase >> (st ^ 1)) & 1u);
            return false;
        }
        phase ^= 1u << st;
        const int cj = cc.cnt;
        const int t0 = cc.k * CHUNK_TILES;

        if (hdr(cc)) {
            // per-block constants: B = q*s split in hi/lo at a per-block
            // exponent E and a per-channel class scale; qz = q.z
            const uint32_t *ksz = reinterpret_cast<const uint32_t *>(stage);
            int Eh[GQ];
            float qzh[GQ];
            {
                float2 xs[GQ][NPAIR];
#pragma unroll
                for (int h = 0; h < GQ; ++h) {
                    float amax = 0.0f;
                    float2 qz2 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int m = 0; m < NPAIR; ++m) {
                        const uint2 sz2 = *reinterpret_cast<const uint2 *>(ksz + 2 * lane + 64 * m);
                        const float2 e0 = __half22float2(*reinterpret_cast<const __half2 *>(&sz2.x));
                        const float2 e1 = __half22float2(*reinterpret_cast<const __half2 *>(&sz2.y));
                        const float2 qv = __half22float2(reinterpret_cast<const __half2 *>(qsm)[(h * D + 2 * lane + 64 * m) / 2]);
                        xs[h][m] = __fmul2_rn(qv, make_float2(e0.x, e1.x));
                        qz2 = __ffma2_rn(qv, make_float2(e0.y, e1.y), qz2);
                        amax = fmaxf(amax, fmaxf(fabsf(xs[h][m].x), fabsf(xs[h][m].y)));
                    }
                    // |x| >= 0 orders like its bits: one warp max-reduce on them
                    amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
                    float qz = qz2.x + qz2.y;
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) qz += __shfl_xor_sync(0xffffffffu, qz, o);
                    const int E = amax > 0.0f ? min(max(14 - (((__float_as_int(amax) >> 23) & 0xff) - 127), -100), 100) : 0;
                    Eh[h] = E;
                    qzh[h] = qz;
                    const float sE = pow2i(E);
#pragma unroll
                    for (int m = 0; m < NPAIR; ++m) {
                        const float sc = sE * clsf[m];
                        const float2 x = __fmul2_rn(xs[h][m], make_float2(sc, sc));
                        const float x0 = x.x, x1 = x.y;
                        const __half2 hi = __floats2half2_rn(x0, x1);
                        const float2 hf = __half22float2(hi);
                        const float2 l2 = __ffma2_rn(hf, make_float2(-1.0f, -1.0f), x);
                        const __half2 lo = __floats2half2_rn(l2.x, l2.y);
                        const int ch = 2 * lane + 64 * m;
                        *reinterpret_cast<__half2 *>(qhl + (h * 2 + 0) * (D + 8) + ch) = hi;
                        *reinterpret_cast<__half2 *>(qhl + (h * 2 + 1) * (D + 8) + ch) = lo;
                    }
                }
                __syncwarp();
                const __half *row = qhl + (hB * 2 + (piece ? 1 : 0)) * (D + 8);
#pragma unroll
                for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
                    for (int o = 0; o < 2; ++o)
                        Bk[kt][o] = *reinterpret_cast<const uint32_t *>(row + 16 * kt + 2 * i + 8 * o);
                __syncwarp();
            }
            // score constants of head hS: logit = raw * c1 + c0 (c1 > 0)
            int Ei = Eh[0];
            float qzi = qzh[0];
#pragma unroll
            for (int h = 1; h < GQ; ++h)
                if (hS == h) { Ei = Eh[h]; qzi = qzh[h]; }
            c1 = pow2i(24 - Ei) * a.sl2;
            c0 = qzi * a.sl2;
        }

        auto body = [&](auto full_tag) {
            constexpr bool FULL = decltype(full_tag)::value;
            const int nt = FULL ? CHUNK_TILES : min(CHUNK_TILES, (cj + TILE - 1) / TILE - t0);
            // phase 1: raw scores of every tile of the chunk (tokens r and
            // r+8, head hS); all tiles' key words are read first so that
            // their unpacking and MMAs interleave
            float sc[CHUNK_TILES][2];
            uint32_t kw[CHUNK_TILES][NW];
#pragma unroll
            for (int tau = 0; tau < CHUNK_TILES; ++tau)
                if (FULL || tau < nt) lds_words<NW>(stage + KSZ + tau * TB + tile_k_off(D) + lane * NW * 4, kw[tau]);
#pragma unroll
            for (int tau = 0; tau < CHUNK_TILES; ++tau) {
                sc[tau][0] = sc[tau][1] = -CUDART_INF_F;
                if (FULL || tau < nt) {
                    uint32_t k10[NW];
#pragma unroll
                    for (int w = 0; w < NW; ++w) k10[w] = kw[tau][w] >> 10;
                    float d4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int kt = 0; kt < NKT; ++kt) {
                        const int q0 = kt, q1 = NKT + kt;
                        const int w0 = 2 * (q0 >> 3), p0 = q0 & 7, w1 = 2 * (q1 >> 3), p1 = q1 & 7;
                        mma16816(d4, ext_rt(kw[tau][w0], k10[w0], p0), ext_rt(kw[tau][w0 + 1], k10[w0 + 1], p0),
                                 ext_rt(kw[tau][w1], k10[w1], p1), ext_rt(kw[tau][w1 + 1], k10[w1 + 1], p1), Bk[kt][0],
                                 Bk[kt][1]);
                    }
                    sc[tau][0] = d4[0] + d4[1];
                    sc[tau][1] = d4[2] + d4[3];
                    if (!FULL) {
                        const int slotk = 16 * (t0 + tau) + r;
                        if (slotk >= cj) sc[tau][0] = -CUDART_INF_F;
                        if (slotk + 8 >= cj) sc[tau][1] = -CUDART_INF_F;
                    }
                }
            }

            // phase 2: running max per head (c1 > 0, so the largest raw
            // score gives the largest logit), rescale on increase
            float mraw = -CUDART_INF_F;
#pragma unroll
            for (int tau = 0; tau < CHUNK_TILES; ++tau) mraw = fmaxf(mraw, fmaxf(sc[tau][0], sc[tau][1]));
            if constexpr (GQ == 1) {
                // every lane scores the one head: a whole-warp max-reduce on
                // order-preserving integer keys (-inf included)
                const int kb = __float_as_int(mraw);
                const int key = __reduce_max_sync(0xffffffffu, kb >= 0 ? kb : kb ^ 0x7fffffff);
                mraw = __int_as_float(key >= 0 ? key : key ^ 0x7fffffff);
            } else {
                mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 4));
                mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 8));
                mraw = fmaxf(mraw, __shfl_xor_sync(0xffffffffu, mraw, 16));
            }
            const float m_new = fmaxf(m_run, fmaf(mraw, c1, c0));
            if (__any_sync(0xffffffffu, m_new > m_run)) {
                const float alpha = m_new > m_run ? ex2(m_run - m_new) : 1.0f;
                l_run *= alpha;
                const float aD = __shfl_sync(0xffffffffu, alpha, 4 * r + i / GPV);
#pragma unroll
                for (int mt = 0; mt < NKT; ++mt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[mt][e] *= aD;
                const float aZ = __shfl_sync(0xffffffffu, alpha, hV);
#pragma unroll
                for (int v = 0; v < NZ; ++v) zs[v] *= aZ;
                zs2 = __fmul2_rn(zs2, make_float2(aZ, aZ));
                m_run = m_new;
            }
            const float c0m = c0 - (m_run == -CUDART_INF_F ? 0.0f : m_run);

            // phase 3a: weights and P' = p*s (hi/lo) for every tile of the chunk
            uint32_t bv[CHUNK_TILES][NV][2];
#pragma unroll
            for (int tau = 0; tau < CHUNK_TILES; ++tau) {
#pragma unroll
                for (int v = 0; v < NV; ++v) bv[tau][v][0] = bv[tau][v][1] = 0u;
                if (FULL || tau < nt) {
                    const uint8_t *tb = stage + KSZ + tau * TB;
                    const float2 lgp = __ffma2_rn(make_float2(sc[tau][0], sc[tau][1]), make_float2(c1, c1),
                                                  make_float2(c0m, c0m));
                    const float p0 = ex2(lgp.x), p1 = ex2(lgp.y);
                    l_run += p0 + p1;
                    if constexpr (SPLIT) {
                        const float pa = __shfl_sync(0xffffffffu, p0, src0);
                        const float pb = __shfl_sync(0xffffffffu, p0, src1);
                        const float pc = __shfl_sync(0xffffffffu, p1, src0);
                        const float pd = __shfl_sync(0xffffffffu, p1, src1);
#pragma unroll
                        for (int k = 0; k < NV / 2; ++k) {
                            // this lane's variant 2k + piece, both pieces; the partner's piece goes across
                            const int gamma = (2 * k + (lo_lane ? 1 : 0)) * GPV + glow;
                            const uint4 sz =
                                *reinterpret_cast<const uint4 *>(tb + tile_sz_off(D) + ((gamma * 4 + i) * 4) * 4);
                            const float2 e0 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.x));
                            const float2 e1 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.y));
                            const float2 e2 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.z));
                            const float2 e3 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.w));
                            const float2 pab = make_float2(pa, pb), pcd = make_float2(pc, pd);
                            const float2 x01 = __fmul2_rn(pab, make_float2(e0.x, e1.x));
                            const float2 x23 = __fmul2_rn(pcd, make_float2(e2.x, e3.x));
                            float2 zk = __fmul2_rn(pab, make_float2(e0.y, e1.y));
                            zk = __ffma2_rn(pcd, make_float2(e2.y, e3.y), zk);
                            zs[k] += zk.x + zk.y;
                            const __half2 h01 = __floats2half2_rn(x01.x, x01.y), h23 = __floats2half2_rn(x23.x, x23.y);
                            const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                            const float2 l01 = __ffma2_rn(f01, make_float2(-1.0f, -1.0f), x01);
                            const float2 l23 = __ffma2_rn(f23, make_float2(-1.0f, -1.0f), x23);
                            const uint32_t hi0 = h2bits(h01), hi1 = h2bits(h23);
                            const uint32_t lo0 = h2bits(__floats2half2_rn(l01.x, l01.y));
                            const uint32_t lo1 = h2bits(__floats2half2_rn(l23.x, l23.y));
                            const uint32_t own0 = lo_lane ? lo0 : hi0, own1 = lo_lane ? lo1 : hi1;
                            const uint32_t got0 = __shfl_xor_sync(0xffffffffu, lo_lane ? hi0 : lo0, 4);
                            const uint32_t got1 = __shfl_xor_sync(0xffffffffu, lo_lane ? hi1 : lo1, 4);
                            bv[tau][2 * k][0] = lo_lane ? got0 : own0;
                            bv[tau][2 * k][1] = lo_lane ? got1 : own1;
                            bv[tau][2 * k + 1][0] = lo_lane ? own0 : got0;
                            bv[tau][2 * k + 1][1] = lo_lane ? own1 : got1;
                        }
                    } else {
                        // one variant: this lane takes tokens 2i, 2i+1 (hi lane) or 2i+8, 2i+9 (lo lane)
                        const float X = send_second ? p1 : p0;
                        const float pA = __shfl_sync(0xffffffffu, X, srcA);
                        const float pB = __shfl_sync(0xffffffffu, X, srcB);
                        const bool gv = glow < NG;           // columns past the value groups stay zero
                        const int gamma = gv ? glow : 0;
                        const uint2 sz = *reinterpret_cast<const uint2 *>(
                            tb + tile_sz_off(D) + (((gamma * 4 + i) * 4) + (lo_lane ? 2 : 0)) * 4);
                        const float2 ea = __half22float2(*reinterpret_cast<const __half2 *>(&sz.x));
                        const float2 eb = __half22float2(*reinterpret_cast<const __half2 *>(&sz.y));
                        const float2 pAB = make_float2(pA, pB);
                        const float2 x = __fmul2_rn(pAB, make_float2(ea.x, eb.x));
                        if (gv) zs2 = __ffma2_rn(pAB, make_float2(ea.y, eb.y), zs2);
                        const __half2 h = __floats2half2_rn(x.x, x.y);
                        const float2 f = __half22float2(h);
                        const float2 l2 = __ffma2_rn(f, make_float2(-1.0f, -1.0f), x);
                        const uint32_t hi = h2bits(h), lo = h2bits(__floats2half2_rn(l2.x, l2.y));
                        // hi lane: keeps hi of (2i, 2i+1), gets hi of (2i+8, 2i+9); lo lane the lo pieces
                        const uint32_t got = __shfl_xor_sync(0xffffffffu, lo_lane ? hi : lo, 4);
                        bv[tau][0][0] = gv ? (lo_lane ? got : hi) : 0u;
                        bv[tau][0][1] = gv ? (lo_lane ? lo : got) : 0u;
                    }
                }
            }
            // phase 3b: the PV products
#pragma unroll
            for (int tau = 0; tau < CHUNK_TILES; ++tau) {
                if (FULL || tau < nt) {
                    uint32_t vw[NW], v10[NW];
                    lds_words<NW>(stage + KSZ + tau * TB + tile_v_off(D) + lane * NW * 4, vw);
#pragma unroll
                    for (int w = 0; w < NW; ++w) v10[w] = vw[w] >> 10;
#pragma unroll
                    for (int mt = 0; mt < NKT; ++mt) {
                        const int q0 = mt, q1 = NKT + mt;
                        const int w0 = 2 * (q0 >> 3), p0_ = q0 & 7, w1 = 2 * (q1 >> 3), p1_ = q1 & 7;
                        const int v = (mt >> 1) / GPV;
                        mma16816(acc[mt], ext_rt(vw[w0], v10[w0], p0_), ext_rt(vw[w1], v10[w1], p1_),
                                 ext_rt(vw[w0 + 1], v10[w0 + 1], p0_), ext_rt(vw[w1 + 1], v10[w1 + 1], p1_),
                                 bv[tau][v][0], bv[tau][v][1]);
                    }
                }
            }
        };
        if (CT * (cc.k + 1) <= cj)
            body(std::true_type{});
        else
            body(std::false_type{});

        // release the stage and refill it with the chunk two ahead
        __syncwarp();
        fence_async_shared();
        if (!past(ic)) {
            issue(ic, st);
            advance(ic);
        }
        advance(cc);
        st ^= 1;
    }

    // epilogue: reduce l over r and the z-sums over i, write the partials
    if constexpr (!SPLIT) zs[0] += zs2.x + zs2.y;
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
    for (int v = 0; v < NZ; ++v) {
        zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], 1);
        zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], 2);
        if constexpr (!SPLIT) zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], 4);   // the pair's tokens
    }
    float *pb = a.part + slot * GQ * (D + 2);
    if (r == 0 && i < GQ) {
        pb[i * (D + 2) + 0] = m_run;
        pb[i * (D + 2) + 1] = l;
    }
    const int hD = i / GPV;
#pragma unroll
    for (int mt = 0; mt < NKT; ++mt) {
        const int gamma = mt >> 1, v = gamma / GPV, gl = gamma % GPV;
        // the lane that summed variant v: piece 0 of its column, or (split) piece v & 1
        const float zval = SPLIT ? __shfl_sync(0xffffffffu, zs[v >> 1], 4 * (2 * (hD * GPV + gl) + (v & 1)))
                                 : __shfl_sync(0xffffffffu, zs[v], 4 * (2 * (hD * GPV + gl)));
        if (gl == i % GPV && hD < GQ) {
            const int ch0 = 16 * mt + r;
            const float sc0 = pow2i(24 - 2 * cls_of_pos(mt & 7));
            const float sc1 = pow2i(24 - 2 * cls_of_pos((NKT + mt) & 7));
            pb[hD * (D + 2) + 2 + ch0] = fmaf(acc[mt][0] + acc[mt][1], sc0, zval);
            pb[hD * (D + 2) + 2 + ch0 + 8] = fmaf(acc[mt][2] + acc[mt][3], sc1, zval);
        }
    }
    return true;
}

// ---------------------------------------------------------------- fp16 segment
// fp16 chunks [c0, c1) of unit u (chunk c = residual-then-pool tokens
// 32c .. 32c+31); the partial goes to part[slot]. Tokens stream through the
// warp's stage ring 8 at a time: one 1-D bulk copy per key and value row into
// rows padded to d+8 halves (conflict-free ldmatrix). Scores: A = key rows
// (ldmatrix), B = q (exact fp16). P.V: A = value rows transposed
// (ldmatrix.trans), B = p split into fp16 hi + lo, mma.sync m16n8k8.
__device__ __forceinline__ void ldsm_x4(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3, const void *p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma1688(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%0,%1,%2,%3};\n"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(b0));
}

// Under the cold-pool policy the fp16 tokens continue with the cold pool
// (token f >= ntail + npool: its (f - ntail - npool)-th oldest entry); its
// size is read on the device, and the host sizes the items for C entries.
template <int D, int GQ, bool CO>
__device__ bool fp16_segment(const DecodeArgs &a, const UnitInfo &ui, size_t slot, int u, int uq, int c0, int c1,
                             uint8_t *stg0, uint8_t *stg1, uint64_t *bars, uint32_t &phase, float *qsm, int lane) {
    constexpr int NKT = D / 16;
    constexpr int RS = D + 8;                 // padded row stride (halves)
    constexpr int SUB = 8;                    // tokens per sub-tile
    const int r = lane >> 2, i = lane & 3;
    int ncold = 0, chead = 0;
    if constexpr (CO) {
        if (a.C > 0) {
            ncold = __ldg(a.cmeta + 2 * u);
            chead = __ldg(a.cmeta + 2 * u + 1);
        }
    }
    const int nhot = ui.ntail + ui.npool, nfp = nhot + ncold;
    const int fb = c0 * FP16_CHUNK, fe = max(fb, min(c1 * FP16_CHUNK, nfp));
    const int nsub = (fe - fb + SUB - 1) / SUB;

    auto row_ptr = [&](int f, bool val) -> const __half * {
        const __half *base = val ? a.rv : a.rk;
        if (f < ui.ntail) {
            int s = ui.ring_start + f;   // f < ntail < ring
            if (s >= a.ring) s -= a.ring;
            return base + ((size_t)u * a.ring + s) * D;
        }
        if constexpr (CO) {
            if (f >= nhot) {
                int s = chead + (f - nhot);   // f - nhot < ncold <= C
                if (s >= a.C) s -= a.C;
                return (val ? a.cv : a.ck) + ((size_t)u * a.C + s) * D;
            }
        }
        return (val ? a.pv : a.pk) + ((size_t)u * a.P + (f - ui.ntail)) * D;
    };
    // lanes 0..7 copy key rows, 8..15 value rows; rows past the end repeat
    // the sub-tile's first token (finite values, masked by a zero weight)
    auto issue = [&](int k, int st) {
        uint8_t *dst = st ? stg1 : stg0;
        if (lane == 0) expect_tx(&bars[st], 2 * SUB * D * 2);
        __syncwarp();
        if (lane < 2 * SUB) {
            const int x = lane & (SUB - 1);
            int f = fb + k * SUB + x;
            if (f >= fe) f = fb + k * SUB;
            bulk_copy_only(dst + (size_t)lane * RS * 2, row_ptr(f, lane >= SUB), D * 2, &bars[st]);
        }
    };
    // the ring and the pool may have been written by the kernel this grid
    // depends on (an append): wait for it before the first copy
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int st_issue = 0;
    for (int k = 0; k < 2 && k < nsub; ++k) {
        issue(k, st_issue);
        st_issue ^= 1;
    }
    load_queries<D, GQ>(a, uq, qsm, lane);
    // score B operand: column r = (head r/2, piece r&1); q is exact in fp16
    const int hB = r >> 1;
    uint32_t Bq[NKT][2];
#pragma unroll
    for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
        for (int o = 0; o < 2; ++o) {
            const __half2 qq = reinterpret_cast<const __half2 *>(qsm)[((hB < GQ ? hB : 0) * D + 16 * kt + 2 * i + 8 * o) / 2];
            Bq[kt][o] = (hB < GQ && (r & 1) == 0) ? h2bits(qq) : 0u;
        }
    float acc[NKT][4];
#pragma unroll
    for (int mt = 0; mt < NKT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    float m_run = -CUDART_INF_F, l_run = 0.0f;   // head i
    const float pm = (r & 1) ? 1.0f : 0.0f;
    const int src0 = 4 * (2 * i) + hB, src1 = 4 * (2 * i + 1) + hB;
    const int lrow = lane & 7, lsel = lane >> 3;   // ldmatrix row provider

    int st = 0;
    for (int k = 0; k < nsub; ++k) {
        const uint8_t *stage = st ? stg1 : stg0;
        if (!mbar_wait(&bars[st], (phase >> st) & 1u)) {
            if (lane == 0) atomicExch(&a.ctl[1], 1);
            mbar_wait(&bars[st ^ 1], (phase >> (st ^ 1)) & 1u);
            return false;
        }
        phase ^= 1u << st;
        const __half *krows = reinterpret_cast<const __half *>(stage);
        const __half *vrows = krows + SUB * RS;
        const int nvalid = min(SUB, fe - (fb + k * SUB));
        // scores: rows 0..7 = tokens (rows 8..15 of the A tile are zero)
        float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int kt = 0; kt < NKT; kt += 2) {
            uint32_t a0, a2, b0, b2;   // (kt, lo), (kt, hi), (kt+1, lo), (kt+1, hi)
            ldsm_x4(a0, a2, b0, b2, krows + lrow * RS + 16 * kt + 8 * lsel);
            mma16816(d, a0, 0u, a2, 0u, Bq[kt][0], Bq[kt][1]);
            mma16816(d, b0, 0u, b2, 0u, Bq[kt + 1][0], Bq[kt + 1][1]);
        }
        float lg = (r < nvalid && i < GQ) ? d[0] * a.sl2 : -CUDART_INF_F;
        float mloc = lg;
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 4));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
        const float m_new = fmaxf(m_run, mloc);
        if (__any_sync(0xffffffffu, m_new > m_run)) {
            const float alpha = m_new > m_run ? ex2(m_run - m_new) : 1.0f;   // head i = this lane's D columns
            l_run *= alpha;
#pragma unroll
            for (int mt = 0; mt < NKT; ++mt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][e] *= alpha;
            m_run = m_new;
        }
        const float pv = ex2(lg - (m_run == -CUDART_INF_F ? 0.0f : m_run));
        l_run += pv;
        // B of P.V: tokens 2i, 2i+1 of head r/2, piece r&1
        const float x0 = __shfl_sync(0xffffffffu, pv, src0), x1 = __shfl_sync(0xffffffffu, pv, src1);
        const __half2 hh = __floats2half2_rn(x0, x1);
        const float2 hf = __half22float2(hh);
        const uint32_t bp = hB < GQ ? h2bits(__floats2half2_rn(x0 - pm * hf.x, x1 - pm * hf.y)) : 0u;
#pragma unroll
        for (int mt = 0; mt < NKT; mt += 2) {
            uint32_t a0, a1, b0, b1;   // channels (mt, lo), (mt, hi), (mt+1, lo), (mt+1, hi)
            ldsm_x4_t(a0, a1, b0, b1, vrows + lrow * RS + 16 * mt + 8 * lsel);
            mma1688(acc[mt], a0, a1, bp);
            mma1688(acc[mt + 1], b0, b1, bp);
        }
        __syncwarp();
        fence_async_shared();
        if (k + 2 < nsub) issue(k + 2, st);
        st ^= 1;
    }
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    float *pb = a.part + slot * GQ * (D + 2);
    if (i < GQ) {
        if (r == 0) {
            pb[i * (D + 2) + 0] = m_run;
            pb[i * (D + 2) + 1] = l;
        }
#pragma unroll
        for (int mt = 0; mt < NKT; ++mt) {
            pb[i * (D + 2) + 2 + 16 * mt + r] = acc[mt][0] + acc[mt][1];
            pb[i * (D + 2) + 2 + 16 * mt + r + 8] = acc[mt][2] + acc[mt][3];
        }
    }
    return true;
}

template <int D, int GQ, bool RG, bool CO, bool TK>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) k_decode(DecodeArgs a, const __grid_constant__ TableT<RG> st) {
    using C = Cfg<D, GQ>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *wbase = smem + (size_t)warp * C::WARP_SMEM;
    uint8_t *stg0 = wbase;
    uint8_t *stg1 = wbase + C::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(wbase + 2 * C::STAGE);
    float *qsm = reinterpret_cast<float *>(wbase + 2 * C::STAGE + 16);
    __half *qhl = reinterpret_cast<__half *>(wbase + 2 * C::STAGE + 16 + GQ * D * 2);
    if (lane == 0) {
        mbar_init(&bars[0]);
        mbar_init(&bars[1]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    // the combine kernel may be scheduled now; it waits for this grid's results
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    uint32_t phase = 0;
    // this warp's contiguous range of work items, split into (unit, type)
    // segments; warp indices are dealt across the CTAs first, so that with
    // fewer active warps than slots every SM still gets its share
    const int gw = warp * gridDim.x + blockIdx.x;
    if (gw >= a.NWp) return;
    // Top-K: launched as a programmatic dependent of the block selection;
    // the selected blocks are that grid's results
    if constexpr (TK) asm volatile("griddepcontrol.wait;" ::: "memory");
    long long x = range_start(a.W, a.NWp, gw);
    const long long x1 = range_start(a.W, a.NWp, gw + 1);
    const int u_first = unit_at<RG>(a, st, x).u;
    while (x < x1) {
        const UnitInfo ui = unit_at<RG>(a, st, x);
        const int u = ui.u;                           // work unit (kv-head slice)
        const int ud = a.S == 1 ? u : u / a.S;        // its kv unit: the cache data
        const long long ubase = ui.ub;
        const int off = (int)(x - ubase);
        if (off < ui.Sf) {
            const int end = (int)min(x1 - ubase, (long long)ui.Sf);
            if (!fp16_segment<D, GQ, CO>(a, ui, part_slot(a, gw, u - u_first, 0), ud, u, off, end, stg0, stg1, bars,
                                     phase, qsm, lane))
                return;
            x = ubase + end;
        } else {
            const int end = (int)min(x1 - ubase, (long long)ui.Iu);
            if (!quant_segment<D, GQ, CO, TK, RG>(a, part_slot(a, gw, u - u_first, 1), ud, u, off - ui.Sf, end - ui.Sf,
                                      stg0, stg1, bars, phase, qsm, qhl, lane))
                return;
            x = ubase + end;
        }
    }
}

// Merge the partials of each (sequence, query head). A CTA of `cw` warps
// serves one (b, hq): the candidate segments of its unit -- (warp, item type)
// pairs of the decode grid whose ranges overlap the unit -- are dealt to the
// warps, each warp folds its share with an online log-sum-exp merge (loads of
// COMB_GRP segments in flight at a time), and warp 0 merges the warps'
// results from shared memory. `cw` is chosen so that each warp needs about
// two rounds: a unit that many decode warps cover (long sequences, few kv
// heads) gets up to 32 combine warps. Launched as a programmatic dependent of
// k_decode: it starts while the decode grid drains and waits for its results.
constexpr int COMB_MAXW = 32;
constexpr int COMB_GRP = 8;     // candidate segments a warp loads at a time

// CS > 1: the channels of a head are split over CS CTAs (each merges every
// partial's max and sum, and its own D/CS channels), so that a batch with
// few query heads still spreads its partials' loads over many SMs.
template <int D, int GQ, bool RG, int CS>
__global__ void __launch_bounds__(COMB_MAXW * 32) k_combine(DecodeArgs a, const __grid_constant__ TableT<RG> st) {
    constexpr int DC = D / CS, CPL = DC / 32, GRP = COMB_GRP;
    static_assert(CPL >= 1, "at least one channel per lane");
    __shared__ float red[COMB_MAXW][DC + 2];
    const int cw = blockDim.x >> 5, wi = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int bh = blockIdx.x / CS, cs = blockIdx.x % CS;
    // work unit of query head hq: kv head hq / g, slice (hq mod g) / GQ
    const int b = bh / a.Hq, hq = bh % a.Hq, hkv = hq / a.g, hs = hq % a.g, h = hs % GQ;
    const int uv = hkv * a.S + hs / GQ, u = b * a.Hkv * a.S + uv;
    const int ch0 = cs * DC + lane * CPL;   // this lane's first channel
    // The unit's items are [ub, ub + Sf) fp16 then [ub + Sf, ue) quantized; the
    // decode warps holding them are contiguous ranges [f0, f1] and [q0, q1].
    // Only the first of them can have started in an earlier unit.
    long long ub;
    int Iu, Sf;
    if constexpr (RG) {
        const SeqEntry &e = st.e[b];
        ub = e.base + (long long)uv * e.Iu;
        Iu = e.Iu;
        Sf = e.Sf;
    } else {
        ub = (long long)u * a.Iu;
        Iu = a.Iu;
        Sf = a.Sf;
    }
    const long long ue = ub + Iu, um = ub + Sf;
    const int wa = warp_of(a.W, a.NWp, ub);
    const int f1 = Sf > 0 ? warp_of(a.W, a.NWp, um - 1) : wa - 1;
    const int q0 = um < ue ? warp_of(a.W, a.NWp, um) : 0, q1 = um < ue ? warp_of(a.W, a.NWp, ue - 1) : -1;
    const int n0 = f1 - wa + 1, ncand = n0 + (q1 - q0 + 1);
    const int uo_a = u - unit_at<RG>(a, st, range_start(a.W, a.NWp, wa)).u;   // unit offset within warp wa's slots
    // everything above depends on the arguments only; the partials are the
    // decode grid's results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // the next decode may be scheduled now (it waits for this grid before
    // reading its inputs or writing partials)
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    float M = -CUDART_INF_F, L = 0.0f, acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.0f;
    for (int k0 = wi * GRP; k0 < ncand; k0 += cw * GRP) {
        // every load of the group is issued before any arithmetic (one round trip)
        float ms[GRP], ls[GRP], vs[GRP][CPL];
#pragma unroll
        for (int g = 0; g < GRP; ++g) {
            ms[g] = -CUDART_INF_F;
            ls[g] = 0.0f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) vs[g][c] = 0.0f;
            const int k = k0 + g;
            if (k < ncand) {
                const int type = k < n0 ? 0 : 1;
                const int ww = type ? q0 + (k - n0) : wa + k;
                const int uo = ww == wa ? uo_a : 0;
                const float *p = a.part + (part_slot(a, ww, uo, type) * GQ + h) * (D + 2);
                ms[g] = p[0];
                ls[g] = p[1];
#pragma unroll
                for (int c = 0; c < CPL; ++c) vs[g][c] = p[2 + ch0 + c];
            }
        }
        float mn = M;
#pragma unroll
        for (int g = 0; g < GRP; ++g) mn = fmaxf(mn, ms[g]);
        if (mn == -CUDART_INF_F) continue;
        const float so = ex2(M - mn);
        L *= so;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] *= so;
#pragma unroll
        for (int g = 0; g < GRP; ++g) {
            const float sn = ex2(ms[g] - mn);   // 0 for an empty segment (m = -inf)
            L = fmaf(sn, ls[g], L);
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(sn, vs[g][c], acc[c]);
        }
        M = mn;
    }
    if (cw > 1) {
        if (lane == 0) {
            red[wi][0] = M;
            red[wi][1] = L;
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) red[wi][2 + lane * CPL + c] = acc[c];
        __syncthreads();
        if (wi != 0) return;
        M = -CUDART_INF_F;
        for (int x = 0; x < cw; ++x) M = fmaxf(M, red[x][0]);
        L = 0.0f;
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = 0.0f;
        for (int x = 0; x < cw; ++x) {
            const float mx = red[x][0];
            if (mx == -CUDART_INF_F) continue;
            const float sx = ex2(mx - M);
            L = fmaf(sx, red[x][1], L);
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[c] = fmaf(sx, red[x][2 + lane * CPL + c], acc[c]);
        }
    }
    __half *o = a.out + ((size_t)b * a.Hq + hq) * D + ch0;
    // one vector store per lane (out may be host memory)
    if constexpr (CPL == 1) {
        *o = __float2half_rn(acc[0] / L);
    } else {
        uint32_t w[CPL / 2];
#pragma unroll
        for (int c = 0; c < CPL; c += 2) w[c / 2] = h2bits(__floats2half2_rn(acc[c] / L, acc[c + 1] / L));
        if constexpr (CPL == 4)
            *reinterpret_cast<uint2 *>(o) = make_uint2(w[0], w[1]);
        else
            *reinterpret_cast<uint32_t *>(o) = w[0];
    }
}

// Launch the combine as a programmatic dependent of the decode grid just
// queued on stream s: one CTA per (sequence, query head).
template <int D, int GQ, bool RG>
cudaError_t launch_combine(const DecodeArgs &a, const TableT<RG> &st, int B, cudaStream_t s) {
    // candidate segments per unit: about 2 * (decode warps covering a unit)
    const long long U = (long long)B * a.Hkv * a.S;
    const long long per_unit_warps = (a.NWp + U - 1) / U + 1;
    int cw = (int)((2 * per_unit_warps + 2 * COMB_GRP - 1) / (2 * COMB_GRP));   // about two rounds per warp
    cw = cw < 1 ? 1 : (cw > COMB_MAXW ? COMB_MAXW : cw);
    // few heads: split their channels so that the CTAs cover the SMs
    const long long heads = (long long)B * a.Hq;
    int cs = 1;
    while (cs < 4 && cs * 2 <= D / 32 && heads * cs * 2 <= 2LL * a.NSM) cs *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(heads * cs));
    cfg.blockDim = dim3((unsigned)(32 * cw));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cs == 4) return cudaLaunchKernelEx(&cfg, k_combine<D, GQ, RG, (D / 32 >= 4 ? 4 : 1)>, a, st);
    if (cs == 2) return cudaLaunchKernelEx(&cfg, k_combine<D, GQ, RG, 2>, a, st);
    return cudaLaunchKernelEx(&cfg, k_combine<D, GQ, RG, 1>, a, st);
}

// One sequence's counts after T tokens and nf flushes.
inline SeqEntry seq_entry(const ott_cache *c, long long T, int nf, int nq_blocks, int ipb) {
    SeqEntry e;
    const long long tail_start = (long long)nf * c->G;
    e.base = 0;
    e.nf = nf;
    e.ring_start = (int)(tail_start % c->ring);
    e.ntail = (int)(T - tail_start);
    e.npool = pool_after(c->P, c->G, nf, c->pct);
    // the cold pool's size is known on the device only: items for all C slots
    const int ncold_max = c->cold > 0 ? c->cold : 0;
    e.Sf = (e.ntail + e.npool + ncold_max + FP16_CHUNK - 1) / FP16_CHUNK;
    e.Iu = e.Sf + nq_blocks * ipb;
    return e;
}

// Kc >= 0: Top-K sparse decode over the Kc selected blocks of every unit.
template <int D, int GQ, bool RG, bool CO, bool TK>
cudaError_t launch_decode_t(const ott_cache *c, const __half *q, __half *out, float *part, cudaStream_t s,
                            int Kc = -1) {
    DecodeArgs a;
    a.sel = c->sel;
    a.Ksel = Kc;
    a.bt = c->paged ? c->bt : nullptr;
    a.bcnt = c->bcnt;
    a.ck = c->ck;
    a.cv = c->cv;
    a.cmeta = c->cmeta;
    a.C = c->cold;
    a.blk = c->blk;
    a.blk_bytes = c->blk_bytes;
    a.NB = c->NB;
    a.rk = c->rk;
    a.rv = c->rv;
    a.ring = c->ring;
    a.pk = c->pk;
    a.pv = c->pv;
    a.P = c->P;
    a.q = q;
    a.out = out;
    a.part = part;
    a.ctl = c->ctl;
    a.Hq = c->Hq;
    a.Hkv = c->Hkv;
    a.g = c->gq;
    a.S = c->S;
    a.G = c->G;
    a.B = c->B;
    a.jfull = (c->P + c->G - 1) / c->G;   // from this block on, the pool is full
    a.CPB = chunks_per_block(c->G);
    // Work items: chunks, so that equal item counts are nearly equal work
    // (the last item of a warp is a small share of it, and per-SM speed
    // differences even out); with fewer blocks than decode warps, whole
    // blocks, so that each warp's fixed cost (queries, block header) is paid
    // once per block.
    long long nblk = 0;
    if constexpr (RG) {
        for (int b = 0; b < c->B; ++b)
            nblk += (long long)c->Hkv * c->S * (TK ? (c->nfb[b] < Kc ? c->nfb[b] : Kc) : c->nfb[b]);
    } else {
        nblk = (long long)c->U * c->S * (TK ? (c->nf < Kc ? c->nf : Kc) : c->nf);
    }
    const long long nwarps = (long long)c->sm_count * DEC_WARPS;
    a.IPB = nblk >= nwarps ? a.CPB : 1;
    TableT<RG> st;
    if constexpr (RG) {
        long long base = 0;
        for (int b = 0; b < c->B; ++b) {
            st.e[b] = seq_entry(c, c->Tb[b], c->nfb[b], TK ? (c->nfb[b] < Kc ? c->nfb[b] : Kc) : c->nfb[b], a.IPB);
            st.e[b].base = base;
            base += (long long)c->Hkv * c->S * st.e[b].Iu;
        }
        st.e[c->B] = SeqEntry{};
        st.e[c->B].base = base;
        a.W = base;
        a.nf = a.ntail = a.npool = a.ring_start = a.Sf = a.Iu = 0;   // per sequence in the table
        a.MAXU = c->maxu_r;
    } else {
        const SeqEntry e = seq_entry(c, c->T, c->nf, TK ? Kc : c->nf, a.IPB);
        a.nf = e.nf;
        a.ring_start = e.ring_start;
        a.ntail = e.ntail;
        a.npool = e.npool;
        a.Sf = e.Sf;
        a.Iu = e.Iu;
        a.W = (long long)c->U * c->S * a.Iu;
        a.MAXU = c->maxu;
    }
    // never more active warps than items: every active warp owns >= 1 item
    a.NWp = (int)(a.W < (long long)c->sm_count * DEC_WARPS ? a.W : (long long)c->sm_count * DEC_WARPS);
    a.sl2 = (float)(1.4426950408889634 / sqrt((double)D));
    a.NSM = c->sm_count;
    // CTAs only as wide as the active warps need: with few items, the SMs keep
    // room for the combine's CTAs, which then start while the decode drains
    const int wpc = (int)(((long long)a.NWp + c->sm_count - 1) / c->sm_count);
    cudaError_t e;
    if constexpr (TK) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)c->sm_count);
        cfg.blockDim = dim3((unsigned)(wpc * 32));
        cfg.dynamicSmemBytes = (size_t)Cfg<D, GQ>::WARP_SMEM * wpc;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, k_decode<D, GQ, RG, CO, TK>, a, st);
    } else {
        // Launched as a programmatic dependent of the kernel before it when
        // no flush was queued since the last decode: its warps then issue
        // their first block copies early and wait for that kernel (an append
        // or the previous call's combine) before reading the queries, the
        // ring, the pool or writing partials. Blocks are written only by
        // flushes, which the host tracks.
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)c->sm_count);
        cfg.blockDim = dim3((unsigned)(wpc * 32));
        cfg.dynamicSmemBytes = (size_t)Cfg<D, GQ>::WARP_SMEM * wpc;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = c->blocks_settled ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, k_decode<D, GQ, RG, CO, TK>, a, st);
    }
    if (e != cudaSuccess) return e;
    return launch_combine<D, GQ, RG>(a, st, c->B, s);
}

template <int D, int GQ>
cudaError_t set_decode_attr(int smem_max) {
    const void *fns[] = {
        reinterpret_cast<const void *>(k_decode<D, GQ, false, false, false>),
        reinterpret_cast<const void *>(k_decode<D, GQ, false, true, false>),
        reinterpret_cast<const void *>(k_decode<D, GQ, true, false, false>),
        reinterpret_cast<const void *>(k_decode<D, GQ, false, false, true>),
        reinterpret_cast<const void *>(k_decode<D, GQ, false, true, true>),
        reinterpret_cast<const void *>(k_decode<D, GQ, true, false, true>),
    };
    for (const void *f : fns) {
        cudaError_t e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

template <int D, int GQ>
cudaError_t launch_decode_any(const ott_cache *c, const __half *q, __half *out, float *part, cudaStream_t s) {
    // block sizes from the per-block counts (cold-pool or channel criterion)
    if (c->bcnt) return launch_decode_t<D, GQ, false, true, false>(c, q, out, part, s);
    return c->ragged ? launch_decode_t<D, GQ, true, false, false>(c, q, out, part, s)
                     : launch_decode_t<D, GQ, false, false, false>(c, q, out, part, s);
}

template <int D, int GQ>
cudaError_t launch_decode_topk_t(const ott_cache *c, const __half *q, __half *out, int Kc, cudaStream_t s) {
    if (c->ragged) return launch_decode_t<D, GQ, true, false, true>(c, q, out, c->part, s, Kc);
    return c->bcnt ? launch_decode_t<D, GQ, false, true, true>(c, q, out, c->part, s, Kc)
                        : launch_decode_t<D, GQ, false, false, true>(c, q, out, c->part, s, Kc);
}

}  // namespace

bool decode_supported(int d) { return d == 64 || d == 128; }

int decode_smem_bytes(int d, int gs) {
#define OTT_SM(D_, G_) \
    if (d == D_ && gs == G_) return Cfg<D_, G_>::WARP_SMEM * DEC_WARPS;
    OTT_SM(128, 1) OTT_SM(128, 2) OTT_SM(128, 4) OTT_SM(64, 1) OTT_SM(64, 2) OTT_SM(64, 4)
#undef OTT_SM
    return 1 << 30;
}

// Both kernels may use up to smem_max bytes of dynamic shared memory (the
// device's opt-in limit), so caches of different shapes never conflict.
cudaError_t set_kernel_attributes(int d, int gs, int smem_max) {
    cudaError_t e = set_flush_attributes(d, smem_max);
    if (e != cudaSuccess) return e;
#define OTT_ATTR(D_, G_) \
    if (d == D_ && gs == G_) return set_decode_attr<D_, G_>(smem_max);
    OTT_ATTR(128, 1) OTT_ATTR(128, 2) OTT_ATTR(128, 4) OTT_ATTR(64, 1) OTT_ATTR(64, 2) OTT_ATTR(64, 4)
#undef OTT_ATTR
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode_topk(const ott_cache *c, const __half *q, __half *out, int Kc, cudaStream_t s) {
#define OTT_DECK(D_, G_) \
    if (c->d == D_ && c->gs == G_) return launch_decode_topk_t<D_, G_>(c, q, out, Kc, s);
    OTT_DECK(128, 1) OTT_DECK(128, 2) OTT_DECK(128, 4) OTT_DECK(64, 1) OTT_DECK(64, 2) OTT_DECK(64, 4)
#undef OTT_DECK
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const ott_cache *c, const __half *q, __half *out, cudaStream_t s) {
#define OTT_DEC(D_, G_) \
    if (c->d == D_ && c->gs == G_) return launch_decode_any<D_, G_>(c, q, out, c->part, s);
    OTT_DEC(128, 1) OTT_DEC(128, 2) OTT_DEC(128, 4) OTT_DEC(64, 1) OTT_DEC(64, 2) OTT_DEC(64, 4)
#undef OTT_DEC
    return cudaErrorInvalidValue;
}

}  // namespace ott

// ---------------------------------------------------------------- diagnostics
namespace ott {
namespace {
__global__ void k_ex2_probe(const float *x, float *y, int n) {
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n; e += gridDim.x * blockDim.x) y[e] = ex2(x[e]);
}
}  // namespace
}  // namespace ott

extern "C" int ott_ex2_probe(const float *x, float *y, int n, void *stream) {
    if (!x || !y || n < 0) return OTT_ERR_INVALID;
    if (n == 0) return OTT_OK;
    const int blocks = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    ott::k_ex2_probe<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y, n);
    return cudaGetLastError() == cudaSuccess ? OTT_OK : OTT_ERR_CUDA;
}

// ---------------------------------------------------------------- allocation-free decode
//
// ott_decode_attn_static: the same two kernels as ott_decode_attn, but the
// split-K partials go to a fixed array in this module's device global memory
// instead of memory the library allocates. It is for callers that may not
// allocate device memory on their decode path: engines that hand all free HBM
// to their own pool at start-up and forbid any later growth, or latency-
// critical loops that cannot afford cudaMalloc's implicit synchronization.
#include <cuda.h>

#include <mutex>

namespace ott {

// 32 MiB of split-K partials, created when a GPU loads this library and held
// by every such GPU until the process exits. All calls share it and it keeps
// the last call's contents; no part of it needs clearing, because a decode
// writes every partial it later reads. Calls that overlap on the GPU (other
// streams, other handles) race on it and must be ordered by the caller.
constexpr size_t kStaticScratchFloats = (size_t)8 << 20;
static __device__ __align__(256) float g_static_scratch[kStaticScratchFloats];

namespace {

std::mutex g_static_mu;
// Host copy of the array's device address per device ordinal, with the id of
// the context it was taken in: after a device reset the module is loaded
// again in a new context, where the array may sit elsewhere, so the address
// is taken again.
struct StaticAddr {
    float *ptr;
    unsigned long long ctx;
};
StaticAddr g_static_addr[1024];

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// The current context's unique id (0 if the driver cannot tell); called
// under g_static_mu.
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static bool resolved = false;
    if (!resolved) {
        void *f1 = nullptr, *f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess && q2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
            get_id = reinterpret_cast<CtxGetIdFn>(f2);
        }
        cudaGetLastError();
        resolved = true;
    }
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx && get_id(ctx, &id) == CUDA_SUCCESS)
        return id;
    return 0;
}

// The array's name is only a host-side stand-in in host code: its device
// address is looked up with the device current, once per device (and again
// in a new context after a device reset).
cudaError_t static_scratch_address(int dev, float **out) {
    if (dev < 0 || dev >= 1024) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_static_mu);
    const unsigned long long ctx = current_context_id();
    StaticAddr &sa = g_static_addr[dev];
    if (!sa.ptr || sa.ctx != ctx) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        sa.ptr = static_cast<float *>(p);
        sa.ctx = ctx;
    }
    *out = sa.ptr;
    return cudaSuccess;
}

}  // namespace
}  // namespace ott

extern "C" int ott_decode_attn_static(ott_cache *c, const void *q, void *out, void *stream) {
    using namespace ott;
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || c->T < 1) return OTT_ERR_STATE;
    if (c->ragged)
        for (int b = 0; b < c->B; ++b)
            if (c->Tb[b] == 0) return OTT_ERR_STATE;   // a released sequence not refilled yet
    if (!q || !out || q == out || (reinterpret_cast<uintptr_t>(q) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u))
        return OTT_ERR_INVALID;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return OTT_ERR_CUDA;
    if (dev != c->device) return OTT_ERR_STATE;   // the cache's device must be current
    const int maxu = c->ragged ? c->maxu_r : c->maxu;
    const size_t need = (size_t)c->sm_count * DEC_WARPS * maxu * 2 * c->gs * (c->d + 2);
    if (need > kStaticScratchFloats) return OTT_ERR_CAPACITY;
    float *scratch = nullptr;
    if (static_scratch_address(dev, &scratch) != cudaSuccess) return OTT_ERR_CUDA;
    cudaError_t e = cudaErrorInvalidValue;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half *qh = static_cast<const __half *>(q);
    __half *oh = static_cast<__half *>(out);
#define OTT_DEC_S(D_, G_) \
    if (c->d == D_ && c->gs == G_) e = launch_decode_any<D_, G_>(c, qh, oh, scratch, s);
    OTT_DEC_S(128, 1) OTT_DEC_S(128, 2) OTT_DEC_S(128, 4) OTT_DEC_S(64, 1) OTT_DEC_S(64, 2) OTT_DEC_S(64, 4)
#undef OTT_DEC_S
    if (e != cudaSuccess) {
        c->poisoned = 1;
        return OTT_ERR_CUDA;
    }
    c->blocks_settled = 1;
    return OTT_OK;
}
