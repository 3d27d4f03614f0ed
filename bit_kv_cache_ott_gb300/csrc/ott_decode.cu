// ott_decode.cu -- decode-step attention over the three OTT stores.
//
// "Accurate KV Cache Quantization with Outlier Tokens Tracing":
// zijie-tian.site sec. 3.3 and the flowchart (the query meets quantized,
// residual-window and outlier keys; the scores are concatenated and
// softmaxed; the weights multiply the matching values and are summed);
// sciencestack.ai Fig. 2 (decoding stage).
//
// Split-K (flash-decoding) design for one GB300:
//   * A persistent grid (one CTA of 8 warps per SM) pulls splits from an
//     atomic counter. A split is a run of quantized blocks of one unit, or
//     32 fp16 tokens (residual ring + pool) of one unit. Every split keeps
//     its own online-softmax state and writes (m, l, acc[d]) per query head;
//     k_combine merges the splits with a log-sum-exp weighting.
//   * Quantized splits: each warp streams its blocks into a private
//     two-stage shared-memory ring with 1-D TMA bulk copies
//     (cp.async.bulk + mbarrier complete_tx), one copy per chunk of up to 8
//     tiles. Waits are bounded; a timeout sets the cache's status word.
//   * Dequantization is folded into the products: q.k_hat =
//     sum_c (q_c s_c) code_c + sum_c q_c z_c and
//     p.v_hat = sum_t (p_t s_t) code_t + sum_t p_t z_t.
//     A code word becomes an fp16x2 mma.sync operand with one AND (the code
//     is an exact fp16 subnormal, see ott_internal.cuh); the other operand
//     (q*s or p*s) is split into fp16 hi + lo for fp32-grade products.
//     Scores: A = K codes [16 tokens x 16 channels], B = q*s [16 x (head,
//     hi/lo)]. PV: A = V codes [16 channels x 16 tokens], B = p*s [16 tokens
//     x (head, group, hi/lo)]. All query heads of a kv head share the codes.
//   * fp16 splits: one lane per token for the scores, one lane per d/32
//     channels for P.V, fp32 accumulation.
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

__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
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
    int nf;
    long long tail_start;
    int ring_start;   // tail_start mod ring
    int ntail, npool;
    int Sq, ipsq, Sf, S_u, total;
    float sl2;   // softmax scale 1/sqrt(d) times log2(e)
};

template <int D, int GQ>
struct Cfg {
    static constexpr int NKT = D / 16;             // score k-tiles = PV m-tiles
    static constexpr int NW = D / 32;              // code words per lane per tile
    static constexpr int NG = D / 32;              // value groups of 32 channels
    static constexpr int GPV = 4 / GQ;             // value groups per PV B variant
    static constexpr int NV = (NG + GPV - 1) / GPV;  // PV B variants
    static constexpr int CPL = D / 32;             // channels per lane, fp16 path
    static constexpr int STAGE = stage_bytes(D);
};

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

// ---------------------------------------------------------------- quantized split
template <int D, int GQ>
__device__ bool quant_split(const DecodeArgs &a, int sg, int u, int j0, int j1, uint8_t *stg0,
                            uint8_t *stg1, uint64_t *bars, uint32_t &phase, float *qsm, int lane) {
    using C = Cfg<D, GQ>;
    constexpr int NKT = C::NKT, NW = C::NW, NG = C::NG, GPV = C::GPV, NV = C::NV;
    constexpr int KSZ = ksz_bytes(D), TB = tile_bytes(D);
    const int r = lane >> 2, i = lane & 3;
    const int b = u / a.Hkv, hkv = u % a.Hkv;
    const int G = a.G, P = a.P;

    float acc[NKT][4];
#pragma unroll
    for (int mt = 0; mt < NKT; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.0f;
    float zs[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) zs[v] = 0.0f;
    float m_run = -CUDART_INF_F, l_run = 0.0f;   // head i
    uint32_t Bk[NKT][2];
    float c1 = 0.0f, c0 = 0.0f;

    // PV B column of this lane: head hV, value-group offset glow, piece
    const int hV = (r >> 1) / GPV, glow = (r >> 1) % GPV;
    const int src0 = 4 * (2 * i) + hV, src1 = 4 * (2 * i + 1) + hV;

    auto active = [&](int j, int k) { return 16 * CHUNK_TILES * k < block_count(P, G, j); };
    int lj = j0, lk = 0;
    while (lj < j1 && !active(lj, lk)) { ++lj; lk = 0; }
    int cj_ = lj, ck_ = lk;   // next chunk to consume

    auto issue = [&](int j, int k, int st) {
        if (lane == 0) {
            const int cj = block_count(P, G, j), vt = (cj + TILE - 1) / TILE;
            const int t0 = k * CHUNK_TILES, nt = min(CHUNK_TILES, vt - t0);
            const uint8_t *bsrc = a.blk + ((size_t)u * a.NB + j) * a.blk_bytes;
            uint8_t *dst = st ? stg1 : stg0;
            if (k == 0)
                bulk_load(dst, bsrc, (uint32_t)(KSZ + nt * TB), &bars[st]);
            else
                bulk_load(dst + KSZ, bsrc + KSZ + (size_t)t0 * TB, (uint32_t)(nt * TB), &bars[st]);
        }
    };
    auto next = [&](int &j, int &k) {
        ++k;
        while (j < j1 && !active(j, k)) { ++j; k = 0; }
    };

    int st_issue = 0;
    for (int n = 0; n < 2 && lj < j1; ++n) {
        issue(lj, lk, st_issue);
        st_issue ^= 1;
        next(lj, lk);
    }
    // the query heads of this kv head, as fp32 in this warp's shared memory
    const int hB = r >> 1;               // score-MMA B column of this lane: head r/2,
    const bool piece = (r & 1) != 0;     // piece r&1 (hi or lo)
    {
        const __half2 *qp = reinterpret_cast<const __half2 *>(a.q + ((size_t)b * a.Hq + hkv * GQ) * D);
        for (int e = lane; e < GQ * D / 2; e += 32) {
            const float2 f = __half22float2(qp[e]);
            qsm[2 * e] = f.x;
            qsm[2 * e + 1] = f.y;
        }
        __syncwarp();
    }
    const float qon = hB < GQ ? 1.0f : 0.0f;
    const float *qrow = qsm + (hB < GQ ? hB : 0) * D;

    int st = 0;
    while (cj_ < j1) {
        uint8_t *stage = st ? stg1 : stg0;
        if (!mbar_wait(&bars[st], (phase >> st) & 1u)) {
            if (lane == 0) atomicExch(&a.ctl[1], 1);
            // let the other copy in flight land before giving up the buffers
            mbar_wait(&bars[st ^ 1], (phase >> (st ^ 1)) & 1u);
            return false;
        }
        phase ^= 1u << st;
        const int cj = block_count(P, G, cj_), vt = (cj + TILE - 1) / TILE;
        const int t0 = ck_ * CHUNK_TILES, nt = min(CHUNK_TILES, vt - t0);

        if (ck_ == 0) {
            // per-block constants: B = q*s split in hi/lo at a class scale
            const uint32_t *ksz = reinterpret_cast<const uint32_t *>(stage);
            float qs[NKT][2][2];
            float amax = 0.0f, qz = 0.0f;
#pragma unroll
            for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    const uint2 sz = *reinterpret_cast<const uint2 *>(ksz + 16 * kt + 2 * i + 8 * o);
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.x));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.y));
                    float2 qq = *reinterpret_cast<const float2 *>(qrow + 16 * kt + 2 * i + 8 * o);
                    qq.x *= qon;
                    qq.y *= qon;
                    qs[kt][o][0] = qq.x * f0.x;
                    qs[kt][o][1] = qq.y * f1.x;
                    qz = fmaf(qq.x, f0.y, qz);
                    qz = fmaf(qq.y, f1.y, qz);
                    amax = fmaxf(amax, fmaxf(fabsf(qs[kt][o][0]), fabsf(qs[kt][o][1])));
                }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            qz += __shfl_xor_sync(0xffffffffu, qz, 1);
            qz += __shfl_xor_sync(0xffffffffu, qz, 2);
            int E = amax > 0.0f ? 14 - (((__float_as_int(amax) >> 23) & 0xff) - 127) : 0;
            E = min(max(E, -100), 100);
            const float pm = piece ? 1.0f : 0.0f;
#pragma unroll
            for (int kt = 0; kt < NKT; ++kt)
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    const int cls = cls_of_pos((o * NKT + kt) & 7);
                    const float sc = pow2i(E - 2 * cls);
                    const float x0 = qs[kt][o][0] * sc, x1 = qs[kt][o][1] * sc;
                    const __half2 hh = __floats2half2_rn(x0, x1);
                    const float2 hf = __half22float2(hh);
                    Bk[kt][o] = h2bits(__floats2half2_rn(x0 - pm * hf.x, x1 - pm * hf.y));
                }
            // score constants of head i (lane 8i holds head i, piece 0)
            const float Ei = __shfl_sync(0xffffffffu, (float)E, 8 * i);
            const float qzi = __shfl_sync(0xffffffffu, qz, 8 * i);
            c1 = pow2i(24 - (int)Ei) * a.sl2;
            c0 = qzi * a.sl2;
        }

        const bool partial = 16 * (t0 + nt) > cj;   // chunk reaches past the valid tokens
        // phase 1: scores of every tile of the chunk (head i, tokens r and r+8)
        float lg[CHUNK_TILES][2];
#pragma unroll
        for (int tau = 0; tau < CHUNK_TILES; ++tau) {
            lg[tau][0] = lg[tau][1] = -CUDART_INF_F;
            if (tau < nt) {
                const uint8_t *tb = stage + KSZ + tau * TB;
                uint32_t kw[NW], k10[NW];
                lds_words<NW>(tb + tile_k_off(D) + lane * NW * 4, kw);
#pragma unroll
                for (int w = 0; w < NW; ++w) k10[w] = kw[w] >> 10;
                float da[4] = {0.0f, 0.0f, 0.0f, 0.0f}, db[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int kt = 0; kt < NKT; ++kt) {
                    const int q0 = kt, q1 = NKT + kt;
                    const int w0 = 2 * (q0 >> 3), p0 = q0 & 7, w1 = 2 * (q1 >> 3), p1 = q1 & 7;
                    mma16816((kt & 1) ? db : da, ext_rt(kw[w0], k10[w0], p0), ext_rt(kw[w0 + 1], k10[w0 + 1], p0),
                             ext_rt(kw[w1], k10[w1], p1), ext_rt(kw[w1 + 1], k10[w1 + 1], p1), Bk[kt][0],
                             Bk[kt][1]);
                }
                const float dsc[4] = {da[0] + db[0], da[1] + db[1], da[2] + db[2], da[3] + db[3]};
                lg[tau][0] = fmaf(dsc[0] + dsc[1], c1, c0);
                lg[tau][1] = fmaf(dsc[2] + dsc[3], c1, c0);
                if (partial) {
                    const int slot = 16 * (t0 + tau) + r;
                    if (slot >= cj) lg[tau][0] = -CUDART_INF_F;
                    if (slot + 8 >= cj) lg[tau][1] = -CUDART_INF_F;
                }
                if (i >= GQ) lg[tau][0] = lg[tau][1] = -CUDART_INF_F;
            }
        }

        // phase 2: running max per head, rescale on increase
        float mloc = -CUDART_INF_F;
#pragma unroll
        for (int tau = 0; tau < CHUNK_TILES; ++tau) mloc = fmaxf(mloc, fmaxf(lg[tau][0], lg[tau][1]));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 4));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 8));
        mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, 16));
        const float m_new = fmaxf(m_run, mloc);
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
            for (int v = 0; v < NV; ++v) zs[v] *= aZ;
            m_run = m_new;
        }
        const float m_use = m_run == -CUDART_INF_F ? 0.0f : m_run;

        // phase 3: weights, P' = p*s (hi/lo) and the PV products
        const float pm = piece ? 1.0f : 0.0f;
#pragma unroll
        for (int tau = 0; tau < CHUNK_TILES; ++tau) {
            if (tau < nt) {
                const uint8_t *tb = stage + KSZ + tau * TB;
                const float p0 = ex2(lg[tau][0] - m_use), p1 = ex2(lg[tau][1] - m_use);
                l_run += p0 + p1;
                const float pa = __shfl_sync(0xffffffffu, p0, src0);
                const float pb = __shfl_sync(0xffffffffu, p0, src1);
                const float pc = __shfl_sync(0xffffffffu, p1, src0);
                const float pd = __shfl_sync(0xffffffffu, p1, src1);
                uint32_t bv[NV][2];
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const int gamma = v * GPV + glow;
                    bv[v][0] = bv[v][1] = 0u;
                    if (gamma < NG) {
                        const uint4 sz =
                            *reinterpret_cast<const uint4 *>(tb + tile_sz_off(D) + ((gamma * 4 + i) * 4) * 4);
                        const float2 e0 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.x));
                        const float2 e1 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.y));
                        const float2 e2 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.z));
                        const float2 e3 = __half22float2(*reinterpret_cast<const __half2 *>(&sz.w));
                        const float x0 = pa * e0.x, x1 = pb * e1.x, x2 = pc * e2.x, x3 = pd * e3.x;
                        zs[v] = fmaf(pa, e0.y, zs[v]);
                        zs[v] = fmaf(pb, e1.y, zs[v]);
                        zs[v] = fmaf(pc, e2.y, zs[v]);
                        zs[v] = fmaf(pd, e3.y, zs[v]);
                        const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
                        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
                        bv[v][0] = h2bits(__floats2half2_rn(x0 - pm * f01.x, x1 - pm * f01.y));
                        bv[v][1] = h2bits(__floats2half2_rn(x2 - pm * f23.x, x3 - pm * f23.y));
                    }
                }
                uint32_t vw[NW], v10[NW];
                lds_words<NW>(tb + tile_v_off(D) + lane * NW * 4, vw);
#pragma unroll
                for (int w = 0; w < NW; ++w) v10[w] = vw[w] >> 10;
#pragma unroll
                for (int mt = 0; mt < NKT; ++mt) {
                    const int q0 = mt, q1 = NKT + mt;
                    const int w0 = 2 * (q0 >> 3), p0_ = q0 & 7, w1 = 2 * (q1 >> 3), p1_ = q1 & 7;
                    const int v = (mt >> 1) / GPV;
                    mma16816(acc[mt], ext_rt(vw[w0], v10[w0], p0_), ext_rt(vw[w1], v10[w1], p1_),
                             ext_rt(vw[w0 + 1], v10[w0 + 1], p0_), ext_rt(vw[w1 + 1], v10[w1 + 1], p1_),
                             bv[v][0], bv[v][1]);
                }
            }
        }

        // release the stage and refill it with the chunk two ahead
        __syncwarp();
        fence_async_shared();
        if (lj < j1) {
            issue(lj, lk, st);
            next(lj, lk);
        }
        next(cj_, ck_);
        st ^= 1;
    }

    // epilogue: reduce l over r and the z-sums over i, write the partials
    float l = l_run;
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
#pragma unroll
    for (int v = 0; v < NV; ++v) {
        zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], 1);
        zs[v] += __shfl_xor_sync(0xffffffffu, zs[v], 2);
    }
    float *pb = a.part + (size_t)sg * GQ * (D + 2);
    if (r == 0 && i < GQ) {
        pb[i * (D + 2) + 0] = m_run;
        pb[i * (D + 2) + 1] = l;
    }
    const int hD = i / GPV;
#pragma unroll
    for (int mt = 0; mt < NKT; ++mt) {
        const int gamma = mt >> 1, v = gamma / GPV, gl = gamma % GPV;
        const float zval = __shfl_sync(0xffffffffu, zs[v], 4 * (2 * (hD * GPV + gl)));
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

// ---------------------------------------------------------------- fp16 split
template <int D, int GQ>
__device__ void fp16_split(const DecodeArgs &a, int sg, int u, int lf, float *qsm, int lane) {
    constexpr int CPL = Cfg<D, GQ>::CPL;
    const int b = u / a.Hkv, hkv = u % a.Hkv;
    const int nfp = a.ntail + a.npool;
    const int f0 = lf * FP16_CHUNK, nvalid = min(FP16_CHUNK, nfp - f0);

    // query heads of this kv head, as fp32 in shared memory
    const __half *qp = a.q + ((size_t)b * a.Hq + hkv * GQ) * D;
    for (int e = lane; e < GQ * D; e += 32) qsm[e] = __half2float(qp[e]);
    __syncwarp();

    auto row_of = [&](int f, const __half *ringb, const __half *poolb) -> const __half * {
        if (f < a.ntail) {
            int slot = a.ring_start + f;   // f < ntail < ring
            if (slot >= a.ring) slot -= a.ring;
            return ringb + ((size_t)u * a.ring + slot) * D;
        }
        return poolb + ((size_t)u * a.P + (f - a.ntail)) * D;
    };

    const bool valid = lane < nvalid;
    float dot[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) dot[h] = 0.0f;
    {
        // the whole key row of this lane's token: all loads in flight at once
        uint4 kv[D / 8];
        const __half *kr = row_of(valid ? f0 + lane : f0, a.rk, a.pk);
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) kv[c8] = valid ? reinterpret_cast<const uint4 *>(kr)[c8] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c8 = 0; c8 < D / 8; ++c8) {
            const __half2 *kh = reinterpret_cast<const __half2 *>(&kv[c8]);
            float kf[8];
#pragma unroll
            for (int x = 0; x < 4; ++x) {
                const float2 f = __half22float2(kh[x]);
                kf[2 * x] = f.x;
                kf[2 * x + 1] = f.y;
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float4 qa = reinterpret_cast<const float4 *>(qsm + h * D + 8 * c8)[0];
                const float4 qb = reinterpret_cast<const float4 *>(qsm + h * D + 8 * c8)[1];
                dot[h] = fmaf(qa.x, kf[0], dot[h]);
                dot[h] = fmaf(qa.y, kf[1], dot[h]);
                dot[h] = fmaf(qa.z, kf[2], dot[h]);
                dot[h] = fmaf(qa.w, kf[3], dot[h]);
                dot[h] = fmaf(qb.x, kf[4], dot[h]);
                dot[h] = fmaf(qb.y, kf[5], dot[h]);
                dot[h] = fmaf(qb.z, kf[6], dot[h]);
                dot[h] = fmaf(qb.w, kf[7], dot[h]);
            }
        }
    }
    float m[GQ], p[GQ], acc[GQ][CPL];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        const float lg = valid ? dot[h] * a.sl2 : -CUDART_INF_F;
        float mx = lg;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        m[h] = mx;
        p[h] = ex2(lg - (mx == -CUDART_INF_F ? 0.0f : mx));
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[h][c] = 0.0f;
    }
    // this lane's channels of the value rows, eight tokens' loads in flight at a time
    using VT = typename std::conditional<CPL == 4, uint2, uint32_t>::type;
#pragma unroll 1
    for (int tb = 0; tb < nvalid; tb += 8) {
        VT vv[8];
#pragma unroll
        for (int x = 0; x < 8; ++x)
            vv[x] = (tb + x < nvalid) ? *reinterpret_cast<const VT *>(row_of(f0 + tb + x, a.rv, a.pv) + lane * CPL)
                                      : VT{};
#pragma unroll
        for (int x = 0; x < 8; ++x) {
            float vf[CPL];
            if constexpr (CPL == 4) {
                const float2 f0_ = __half22float2(*reinterpret_cast<const __half2 *>(&vv[x].x));
                const float2 f1_ = __half22float2(*reinterpret_cast<const __half2 *>(&vv[x].y));
                vf[0] = f0_.x; vf[1] = f0_.y; vf[2] = f1_.x; vf[3] = f1_.y;
            } else {
                const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&vv[x]));
                vf[0] = f.x; vf[1] = f.y;
            }
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                const float pt = __shfl_sync(0xffffffffu, p[h], (tb + x) & 31);
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc[h][c] = fmaf(pt, vf[c], acc[h][c]);
            }
        }
    }
    float *pb = a.part + (size_t)sg * GQ * (D + 2);
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float l = p[h];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            pb[h * (D + 2) + 0] = m[h];
            pb[h * (D + 2) + 1] = l;
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c) pb[h * (D + 2) + 2 + lane * CPL + c] = acc[h][c];
    }
    __syncwarp();
}

template <int D, int GQ>
__global__ void __launch_bounds__(DEC_WARPS * 32, 1) k_decode(DecodeArgs a) {
    using C = Cfg<D, GQ>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *stg0 = smem + (size_t)warp * 2 * C::STAGE;
    uint8_t *stg1 = stg0 + C::STAGE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)DEC_WARPS * 2 * C::STAGE) + 2 * warp;
    float *qsm = reinterpret_cast<float *>(smem + (size_t)DEC_WARPS * 2 * C::STAGE + DEC_WARPS * 16) +
                 (size_t)warp * GQ * D;
    if (lane == 0) {
        mbar_init(&bars[0]);
        mbar_init(&bars[1]);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    uint32_t phase = 0;
    // the next split's id is fetched one split ahead, so the atomic's round
    // trip overlaps the current split
    int s_next = 0;
    if (lane == 0) s_next = atomicAdd(&a.ctl[0], 1);
    s_next = __shfl_sync(0xffffffffu, s_next, 0);
    while (s_next < a.total) {
        const int s = s_next;
        if (lane == 0) s_next = atomicAdd(&a.ctl[0], 1);
        s_next = __shfl_sync(0xffffffffu, s_next, 0);
        const int u = s / a.S_u, ls = s % a.S_u;
        if (ls < a.Sq) {
            if (!quant_split<D, GQ>(a, s, u, ls * a.ipsq, min(a.nf, (ls + 1) * a.ipsq), stg0, stg1, bars,
                                    phase, qsm, lane))
                break;
        } else {
            fp16_split<D, GQ>(a, s, u, ls - a.Sq, qsm, lane);
        }
    }
}

template <int D, int GQ>
__global__ void k_combine(const float *__restrict__ part, __half *__restrict__ out, int *ctl, int B, int Hq,
                          int Hkv, int S_u) {
    constexpr int CPL = D / 32;
    if (blockIdx.x == 0 && threadIdx.x == 0) ctl[0] = 0;   // re-arm the split counter
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= B * Hq) return;
    const int b = w / Hq, hq = w % Hq, u = b * Hkv + hq / GQ, h = hq % GQ;
    const size_t sstride = (size_t)GQ * (D + 2);
    const float *base = part + ((size_t)u * S_u * GQ + h) * (D + 2);
    float M = -CUDART_INF_F;
    for (int s = lane; s < S_u; s += 32) M = fmaxf(M, base[s * sstride]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.0f, acc[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) acc[c] = 0.0f;
    for (int s = 0; s < S_u; ++s) {
        const float *ps = base + s * sstride;
        const float ms = ps[0];
        const float wgt = ms == -CUDART_INF_F ? 0.0f : exp2f(ms - M);
        L = fmaf(wgt, ps[1], L);
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = fmaf(wgt, ps[2 + lane * CPL + c], acc[c]);
    }
    __half *o = out + ((size_t)b * Hq + hq) * D + lane * CPL;
#pragma unroll
    for (int c = 0; c < CPL; ++c) o[c] = __float2half_rn(acc[c] / L);
}

template <int D, int GQ>
cudaError_t launch_decode_t(const ott_cache *c, const __half *q, __half *out, cudaStream_t s) {
    DecodeArgs a;
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
    a.part = c->part;
    a.ctl = c->ctl;
    a.Hq = c->Hq;
    a.Hkv = c->Hkv;
    a.G = c->G;
    a.nf = c->nf;
    a.tail_start = (long long)c->nf * c->G;
    a.ring_start = (int)(a.tail_start % c->ring);
    a.ntail = (int)(c->T - a.tail_start);
    a.npool = pool_after(c->P, c->G, c->nf);
    const int nfp = a.ntail + a.npool;
    a.Sf = (nfp + FP16_CHUNK - 1) / FP16_CHUNK;
    // blocks per quantized split: aim at ~8 splits per resident warp overall
    const long long target = 8LL * c->sm_count * DEC_WARPS;
    const long long per_unit = target / c->U > 1 ? target / c->U : 1;
    int ipsq = c->nf > 0 ? (int)((c->nf + per_unit - 1) / per_unit) : 1;
    ipsq = ipsq < 1 ? 1 : (ipsq > 4 ? 4 : ipsq);
    a.Sq = (c->nf + ipsq - 1) / ipsq;
    while (a.Sq + a.Sf > c->su_max) {   // split capacity of the scratch buffer
        ++ipsq;
        a.Sq = (c->nf + ipsq - 1) / ipsq;
    }
    a.ipsq = ipsq;
    a.S_u = a.Sq + a.Sf;
    a.total = c->U * a.S_u;
    a.sl2 = (float)(1.4426950408889634 / sqrt((double)D));
    const int smem = decode_smem_bytes(D, GQ);
    k_decode<D, GQ><<<c->sm_count, DEC_WARPS * 32, smem, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int warps = c->B * c->Hq, th = 256, bl = (warps * 32 + th - 1) / th;
    k_combine<D, GQ><<<bl, th, 0, s>>>(c->part, out, c->ctl, c->B, c->Hq, c->Hkv, a.S_u);
    return cudaGetLastError();
}

template <int D, int GQ>
cudaError_t set_decode_attr(int smem_max) {
    return cudaFuncSetAttribute(k_decode<D, GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
}

}  // namespace

bool decode_supported(int d, int gq) {
    return (d == 64 || d == 128) && (gq == 1 || gq == 2 || gq == 4);
}

int decode_smem_bytes(int d, int gq) {
    return DEC_WARPS * (2 * stage_bytes(d) + 16 + gq * d * 4);
}

// Both kernels may use up to smem_max bytes of dynamic shared memory (the
// device's opt-in limit), so caches of different shapes never conflict.
cudaError_t set_kernel_attributes(int d, int gq, int smem_max) {
    cudaError_t e = set_flush_attributes(d, smem_max);
    if (e != cudaSuccess) return e;
#define OTT_ATTR(D_, G_) \
    if (d == D_ && gq == G_) return set_decode_attr<D_, G_>(smem_max);
    OTT_ATTR(128, 1) OTT_ATTR(128, 2) OTT_ATTR(128, 4) OTT_ATTR(64, 1) OTT_ATTR(64, 2) OTT_ATTR(64, 4)
#undef OTT_ATTR
    return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const ott_cache *c, const __half *q, __half *out, cudaStream_t s) {
#define OTT_DEC(D_, G_) \
    if (c->d == D_ && c->gq == G_) return launch_decode_t<D_, G_>(c, q, out, s);
    OTT_DEC(128, 1) OTT_DEC(128, 2) OTT_DEC(128, 4) OTT_DEC(64, 1) OTT_DEC(64, 2) OTT_DEC(64, 4)
#undef OTT_DEC
    return cudaErrorInvalidValue;
}

}  // namespace ott
