// ott_flush.cu -- append, flush (norm, top-P pool merge, 2-bit quantization,
// packing), prefill tail copy and the canonical state export.
//
// The flush follows "Accurate KV Cache Quantization with Outlier Tokens
// Tracing": zijie-tian.site sec. 3.1 (every G tokens the oldest group is
// quantized; candidates are ranked by the key norm) and sec. 3.2 (an outlier
// pool of capacity P; new tokens compete with the pool; a displaced token is
// written back to the quantized cache); sciencestack.ai Abstract (keys per
// channel, values per token) and Fig. 1(c) (keep the smallest-magnitude keys).
//
// One CTA per unit (sequence, kv head). The candidates (pool + group) are
// staged in shared memory; the squared norm of each group key is summed in
// fp32 in channel order; every candidate's rank under (norm, token index) is
// counted; the P best stay (pool slot = rank), the rest form the block in
// ascending token order. Keys are quantized per channel, values per token per
// 32 channels, with IEEE fp32 steps (__fsub_rn/__fdiv_rn, round-half-even
// __float2int_rn) and fp16 round-to-nearest for scale and zero.
//
// Cold-pool policy (zijie-tian.site sec. 3.2, the alternative to writing a
// displaced token back): the displaced pool tokens do not join the block;
// they enter the unit's cold pool, an fp16 ring of C slots used first in,
// first out, in ascending token order, and the tokens that entered first are
// discarded when it overflows. The block is then the group's tokens that did
// not enter the pool, and its size, which depends on the data, is written to
// the per-block count array.
#include <math_constants.h>

#include <algorithm>
#include <climits>

#include "ott_internal.cuh"

namespace ott {
namespace {

constexpr int FLUSH_THREADS = 512;

// The 2-bit code of x under scale s and zero z is clamp(rint(fl((x - z) / s)),
// 0, 3) with fp32 round-to-nearest-even division and rint. Writing
// f = fl(y), y = (x - z) / s and a = fl(x - z), the code is
// [f > 1/2] + [f >= 3/2] + [f > 5/2]; fp32 rounding is monotone and 1/2, 3/2,
// 5/2 have even significands (a tie at a midpoint rounds onto them), so
//   f > 1/2  <=>  y > 1/2 + 2^-25  <=>  a > RD(s (1/2 + 2^-25))
//   f >= 3/2 <=>  y >= 3/2 - 2^-24 <=>  a >= RU(s (3/2 - 2^-24))
//   f > 5/2  <=>  y > 5/2 + 2^-23  <=>  a > RD(s (5/2 + 2^-23))
// (a is an fp32 value, so comparing it with a real c is comparing it with c
// rounded down, or up for >=). The scales are fp16 values (11 significant
// bits, >= 2^-24), so s/2, 3s/2, 5s/2 and s 2^-k are exact in fp32 and each
// threshold is one directed-rounding add of two exact terms. Code = three
// compares instead of a division; the same codes bit for bit.
__device__ __forceinline__ float4 code_rule(float s, float z) {
    if (s == 0.0f) return make_float4(z, CUDART_INF_F, CUDART_INF_F, CUDART_INF_F);   // every code 0
    const float t1 = __fadd_rd(__fmul_rn(0.5f, s), __fmul_rn(s, 0x1p-25f));
    const float t2 = __fsub_ru(__fmul_rn(1.5f, s), __fmul_rn(s, 0x1p-24f));
    const float t3 = __fadd_rd(__fmul_rn(2.5f, s), __fmul_rn(s, 0x1p-23f));
    return make_float4(z, t1, t2, t3);
}

// fl32(x - z) for the fp16 value in the low (hi = 0) or high half of w: the
// mixed-precision subtraction converts x exactly and rounds once
__device__ __forceinline__ float sub_h(uint32_t w, bool hi, float z) {
    float d;
    if (hi)
        asm("{ .reg .f16 l, h;\n mov.b32 {l, h}, %1;\n sub.rn.f32.f16 %0, h, %2; }" : "=f"(d) : "r"(w), "f"(z));
    else
        asm("{ .reg .f16 l, h;\n mov.b32 {l, h}, %1;\n sub.rn.f32.f16 %0, l, %2; }" : "=f"(d) : "r"(w), "f"(z));
    return d;
}
// the code of a = fl32(x - z) under the rule r = (z, t1, t2, t3)
__device__ __forceinline__ uint32_t qcode_a(float a, const float4 &r) {
    return (uint32_t)(a > r.y) + (uint32_t)(a >= r.z) + (uint32_t)(a > r.w);
}
// s + x*x for the fp16 value in half `hi` of w, one rounding (x*x is exact in fp32)
__device__ __forceinline__ float sq_acc(uint32_t w, bool hi, float s) {
    float d;
    if (hi)
        asm("{ .reg .f16 l, h;\n mov.b32 {l, h}, %1;\n fma.rn.f32.f16 %0, h, h, %2; }" : "=f"(d) : "r"(w), "f"(s));
    else
        asm("{ .reg .f16 l, h;\n mov.b32 {l, h}, %1;\n fma.rn.f32.f16 %0, l, l, %2; }" : "=f"(d) : "r"(w), "f"(s));
    return d;
}

__device__ __forceinline__ void cp_async8(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem_dst)), "l"(gsrc) : "memory");
}
// 16 bytes, cached in L2 only (each row is read once)
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
// wait until at most N of this thread's committed groups are still in flight
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// Position of channel ch within staged row r: the row's 16-byte chunks are
// permuted by XOR with r mod 8.
__device__ __forceinline__ int SWZ(int r, int ch) { return (((ch >> 3) ^ (r & 7)) << 3) | (ch & 7); }

// Staged-row layout: padded rows (stride D + 8 halves, no address
// arithmetic) or unpadded swizzled rows (stride D, chunk index XOR r mod 8),
// which save 16 bytes per row where the padding would cost a second CTA per
// SM.
template <int D, bool SW>
struct Rows {
    static constexpr int RS = SW ? D : D + 8;
    __device__ static __forceinline__ int pos(int r, int ch) { return SW ? SWZ(r, ch) : ch; }
    __device__ static __forceinline__ int chunk(int r, int v8) { return SW ? (v8 ^ (r & 7)) : v8; }
};

// Two fp16 values (bit patterns, one per 16-bit lane) -> 16-bit signed keys
// in the values' order, with -0 below +0 (so that min and max do not depend
// on the order the values come in): a negative value keeps its sign bit and
// has its magnitude bits flipped. The map is its own inverse.
__device__ __forceinline__ uint32_t okey2(uint32_t h2) {
    // 0xffff in each 16-bit lane whose sign bit is set (byte permute with
    // sign replication of bytes 1 and 3)
    uint32_t m;
    asm("prmt.b32 %0, %1, %2, 0xBB99;" : "=r"(m) : "r"(h2), "r"(0u));
    return h2 ^ (m & 0x7fff7fffu);
}
// the fp16 value of the key in the low 16-bit lane
__device__ __forceinline__ float okey_lo(uint32_t k2) {
    return __half2float(__ushort_as_half((unsigned short)(okey2(k2) & 0xffffu)));
}

__device__ __forceinline__ uint32_t half2_bits(__half a, __half b) {
    return (uint32_t)__half_as_ushort(a) | ((uint32_t)__half_as_ushort(b) << 16);
}

struct FlushArgs {
    uint8_t *blk;
    int32_t *bidx;
    __half *pk, *pv;
    float *pnorm;
    int32_t *pidx;
    const __half *srcK, *srcV;
    __half *ck, *cv;             // cold pool [U][C][d] (cold-pool policy)
    int32_t *cidx;               // [U][C] token index of each cold slot
    int *cmeta;                  // [U][2]: tokens in the cold pool, slot of the oldest
    int32_t *bcnt;               // [U][NB] valid tokens of each block (null: fixed by P, G, j)
    int C;                       // cold-pool capacity; -1: displaced tokens are written back
    int pct, n_oc;               // channel-conditioned criterion: p (1/10000; -1: norm) and channels
    int32_t *bt;                 // paged pool: [U][NB] slot of each block (null: slot u*NB + j)
    int32_t *fstack;             // paged pool: free slots
    int *ftop;                   // paged pool: number of free slots
    int *ctl;                    // status word: [1] set when the pool had no free slot
    // parallel prefill: every flush of units [pf_u0, pf_u0 + nu) in one
    // launch (CTA i: unit pf_u0 + i / pf_nf, group i % pf_nf); the pool
    // before group j is read from the pool history (keys of the pool after
    // flush j - 1, ascending) and its rows from the prefill source
    const uint64_t *phist;       // [nu][pf_nf][P], or null
    int pf_nf, pf_u0;
    int src_u0;                  // the source holds units src_u0, src_u0 + 1, ...
    long long src_unit_stride;   // elements between units in the source
    long long src_mod;           // slot = token mod src_mod
    long long t0;                // first token of the group
    long long blk_bytes;
    int G, P, NB, ntile, j, np0;
    int Hkv;
};

// One CTA per unit. Without a list, CTA u flushes group a.j of unit u; with
// one (ragged batches), CTA i flushes group fl.lj[i / Hkv] of kv head i % Hkv
// of sequence fl.lb[i / Hkv].
template <int D, bool SW>
__global__ void __launch_bounds__(FLUSH_THREADS, 2) k_flush(FlushArgs a, const __grid_constant__ FlushList fl) {
    extern __shared__ __align__(16) uint8_t smem[];
    // Staged rows are D halves, unpadded; the 16-byte chunks of row r are
    // permuted by XOR with r mod 8 (SWZ), so that the same chunk of 8
    // consecutive rows falls on 8 different bank groups.
    constexpr int VPR = D / 8;         // 16-byte vectors per row
    constexpr int NG = D / 32;         // value groups
    constexpr int NKT = D / 16;
    constexpr int NW = D / 32;
    const int tid = threadIdx.x, nth = blockDim.x;
    int u = blockIdx.x, jj = a.j;
    long long t0 = a.t0;
    const uint64_t *ph = nullptr;      // parallel prefill: the pool before this group
    if (a.phist) {
        u = a.pf_u0 + blockIdx.x / a.pf_nf;
        jj = blockIdx.x % a.pf_nf;
        t0 = (long long)jj * a.G;
        if (jj > 0) ph = a.phist + ((size_t)(u - a.pf_u0) * a.pf_nf + (jj - 1)) * a.P;
    } else if (fl.n > 0) {
        const int e = blockIdx.x / a.Hkv;
        u = fl.lb[e] * a.Hkv + blockIdx.x % a.Hkv;
        jj = fl.lj[e];
        t0 = (long long)jj * a.G;
    }
    const int G = a.G, P = a.P;
    const int np0 = (a.phist || fl.n > 0) ? pool_after(P, G, jj, a.pct) : a.np0, nc = np0 + G;

    __half *ck = reinterpret_cast<__half *>(smem);
    using RL = Rows<D, SW>;
    constexpr int RS = RL::RS;
    __half *cv = ck + (size_t)nc * RS;
    uint64_t *key = reinterpret_cast<uint64_t *>(cv + (size_t)nc * RS);
    int *rank = reinterpret_cast<int *>(key + nc);
    int *bmap = rank + nc;
    int *emap = bmap + G;              // displaced pool rows by token order (cold-pool policy)
    // code rules: per channel for keys, per (token, 32 channels) for values;
    // the value area first holds the key min/max partials
    const size_t rule_off = ((size_t)(reinterpret_cast<uint8_t *>(emap + (P > 0 ? P : 1)) - smem) + 15) & ~(size_t)15;
    // Rule arrays are skewed by one entry per 8 so that the pack phase's
    // loads (8 channels or 8 tokens, 2 apart, per warp) hit distinct banks:
    // channel ch at krule[ch + ch/8]; token t of value group g at
    // vrule[g*VS + t + t/8].
    float4 *krule = reinterpret_cast<float4 *>(smem + rule_off);
    float4 *vrule = krule + D + D / 8;
    const int TS = a.ntile * TILE, VS = TS + TS / 8;
    float *ks = reinterpret_cast<float *>(krule);   // channel criterion scratch (before the rules)
    float *kz = ks + D;
    const int warp = tid >> 5, lane = tid & 31, nwarp = nth >> 5;

    // 1. stage the candidates: old pool rows, then the group's rows, by
    // asynchronous 16-byte copies (every thread's loads in flight at once).
    // Source slots: token t sits at t mod src_mod (the ring wraps; a prompt
    // does not). The group's tokens are consecutive, so their slots follow
    // from the first one with at most one wrap (G <= the ring).
    {
        const size_t uoff = (size_t)(u - a.src_u0) * a.src_unit_stride;
        const __half *srcK = a.srcK + uoff, *srcV = a.srcV + uoff;
        const long long s0 = t0 % a.src_mod;
        for (int e = tid; e < nc * VPR; e += nth) {
            const int row = e / VPR, v8 = e % VPR;
            const __half *sk, *sv;
            if (row < np0 && !ph) {
                const size_t off = ((size_t)u * P + row) * D;
                sk = a.pk + off;
                sv = a.pv + off;
            } else {
                long long slot;
                if (row < np0) {
                    slot = (long long)(uint32_t)ph[row];
                    if (slot >= a.src_mod) slot %= a.src_mod;
                } else {
                    slot = s0 + (row - np0);
                    if (slot >= a.src_mod) slot -= a.src_mod;
                }
                sk = srcK + (size_t)slot * D;
                sv = srcV + (size_t)slot * D;
            }
            cp_async16(reinterpret_cast<uint4 *>(ck + (size_t)row * RS) + RL::chunk(row, v8),
                       reinterpret_cast<const uint4 *>(sk) + v8);
            cp_async16(reinterpret_cast<uint4 *>(cv + (size_t)row * RS) + RL::chunk(row, v8),
                       reinterpret_cast<const uint4 *>(sv) + v8);
        }
    }
    cp_async_wait_all();
    __syncthreads();

    // 2. keys: (fp32 squared norm bits, token index); norms >= +0 order as bits
    const bool chan = a.pct >= 0;
    if (!chan) {
        for (int row = tid; row < nc; row += nth) {
            float nrm;
            int idx;
            if (row < np0 && ph) {
                key[row] = ph[row];
                continue;
            }
            if (row < np0) {
                nrm = a.pnorm[(size_t)u * P + row];
                idx = a.pidx[(size_t)u * P + row];
            } else {
                const uint4 *kr = reinterpret_cast<const uint4 *>(ck + (size_t)row * RS);
                float s = 0.0f;
                for (int v8 = 0; v8 < VPR; ++v8) {   // channels 8 v8 .. 8 v8 + 7, in order
                    const uint4 x = kr[RL::chunk(row, v8)];
                    const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        s = sq_acc(w4[e], false, s);
                        s = sq_acc(w4[e], true, s);
                    }
                }
                nrm = s;
                idx = (int)(t0 + (row - np0));
            }
            key[row] = ((uint64_t)__float_as_uint(nrm) << 32) | (uint32_t)idx;
        }
    } else {
        // channel-conditioned criterion: the outlier channels are the n_oc
        // with the largest max |k| over all candidates (ties to the lower
        // channel); every candidate, old pool rows included, is scored by
        // its squared norm over them (fp32, ascending channel order).
        // ks and kz are free until step 6.
        float *camax = ks;
        int *csel = reinterpret_cast<int *>(kz);
        for (int ch = tid; ch < D; ch += nth) {
            float m = 0.0f;
            for (int row = 0; row < nc; ++row) m = fmaxf(m, fabsf(__half2float(ck[(size_t)row * RS + RL::pos(row, ch)])));
            camax[ch] = m;
        }
        __syncthreads();
        for (int ch = tid; ch < D; ch += nth) {
            const float m = camax[ch];
            int rk = 0;
            for (int c2 = 0; c2 < D; ++c2) rk += camax[c2] > m || (camax[c2] == m && c2 < ch);
            csel[ch] = rk < a.n_oc;
        }
        __syncthreads();
        for (int row = tid; row < nc; row += nth) {
            const __half *kr = ck + (size_t)row * RS;
            float s = 0.0f;
            for (int ch = 0; ch < D; ++ch) {
                if (!csel[ch]) continue;
                const float x = __half2float(kr[RL::pos(row, ch)]);
                s = __fadd_rn(s, __fmul_rn(x, x));
            }
            const int idx = row < np0 ? a.pidx[(size_t)u * P + row] : (int)(t0 + (row - np0));
            key[row] = ((uint64_t)__float_as_uint(s) << 32) | (uint32_t)idx;
        }
    }
    __syncthreads();

    // 3. rank of every candidate under (norm, index); keys are distinct.
    // Each candidate's count is split into `parts` ranges of the others,
    // summed by shared-memory atomics.
    for (int r = tid; r < nc; r += nth) rank[r] = 0;
    __syncthreads();
    {
        const int parts = nc < nth ? nth / nc : 1;
        for (int e = tid; e < nc * parts; e += nth) {
            const int r = e % nc, part = e / nc;
            const int q0 = (nc * part) / parts, q1 = (nc * (part + 1)) / parts;
            const uint64_t kr = key[r];
            int c = 0;
            for (int q = q0; q < q1; ++q) c += key[q] < kr;
            if (c) atomicAdd(rank + r, c);
        }
    }
    __syncthreads();
    // the pool keeps the P best, or under the channel criterion at most the
    // ceil(p * nc) smallest scores
    int keep = min(P, nc);
    if (chan) keep = min(keep, (int)(((long long)a.pct * nc + 9999) / 10000));
    const bool cold = a.C >= 0;
    // pool tokens that leave the pool (every warp counts them by ballots);
    // under the cold-pool policy they also leave the block
    int nlp = 0;
    for (int q0 = 0; q0 < np0; q0 += 32) {
        const int q = q0 + lane;
        nlp += __popc(__ballot_sync(0xffffffffu, q < np0 && rank[q] >= keep));
    }
    const int ev = cold ? nlp : 0;
    const int cnt = nc - keep - ev;

    // 4. block slot of every leaving candidate (cold-pool policy: of every
    // leaving group token, and cold order of every displaced pool token):
    // rank by token index among its own kind
    // Every pool token precedes every group token, and the group rows are
    // staged in token order: a leaving group row's place is the leaving pool
    // tokens (written back ones only) plus the leaving group rows before it,
    // a prefix count taken by warp ballots over chunks of 32 rows.
    for (int c = warp; c < (G + 31) / 32; c += nwarp) {
        int base = cold ? 0 : nlp;
        for (int k = 0; k < c; ++k) {
            const int g = 32 * k + lane;
            base += __popc(__ballot_sync(0xffffffffu, g < G && rank[np0 + g] >= keep));
        }
        const int g = 32 * c + lane;
        const bool f = g < G && rank[np0 + g] >= keep;
        const uint32_t bal = __ballot_sync(0xffffffffu, f);
        if (f) bmap[base + __popc(bal & ((1u << lane) - 1u))] = np0 + g;
    }
    // a leaving pool row: its place among the leaving pool rows by token index
    for (int r = tid; r < np0; r += nth) {
        if (rank[r] < keep) continue;
        const uint32_t ir = (uint32_t)key[r];
        int pos = 0;
        for (int q = 0; q < np0; ++q) pos += (rank[q] >= keep) && ((uint32_t)key[q] < ir);
        if (cold)
            emap[pos] = r;
        else
            bmap[pos] = r;
    }
    // cold pool before this flush (read by every thread before thread 0
    // updates it below)
    int cn0 = 0, ch0 = 0;
    if (cold && a.C > 0) {
        cn0 = a.cmeta[2 * u];
        ch0 = a.cmeta[2 * u + 1];
    }
    // 5. the new pool (old pool rows are already staged in shared memory);
    // a parallel prefill keeps only the last group's
    const bool write_pool = !a.phist || jj == a.pf_nf - 1;
    {
        uint4 *pk_u = reinterpret_cast<uint4 *>(a.pk + (size_t)u * P * D);
        uint4 *pv_u = reinterpret_cast<uint4 *>(a.pv + (size_t)u * P * D);
        for (int e = tid; write_pool && e < nc * VPR; e += nth) {
            const int row = e / VPR, v8 = e % VPR, rk = rank[row];
            if (rk < keep) {
                pk_u[rk * VPR + v8] = reinterpret_cast<const uint4 *>(ck + (size_t)row * RS)[RL::chunk(row, v8)];
                pv_u[rk * VPR + v8] = reinterpret_cast<const uint4 *>(cv + (size_t)row * RS)[RL::chunk(row, v8)];
            }
        }
    }
    for (int row = tid; write_pool && row < nc; row += nth) {
        const int rk = rank[row];
        if (rk < keep) {
            a.pnorm[(size_t)u * P + rk] = __uint_as_float((uint32_t)(key[row] >> 32));
            a.pidx[(size_t)u * P + rk] = (int32_t)(uint32_t)key[row];
        }
    }
    __syncthreads();

    // the displaced tokens enter the cold pool in token order; of the
    // cn0 + ev tokens, the last min(C, cn0 + ev) stay
    if (a.bcnt && tid == 0) a.bcnt[(size_t)u * a.NB + jj] = cnt;
    if (cold) {
        if (a.C > 0 && ev > 0) {
            const int n1 = min(a.C, cn0 + ev), skip = ev - min(ev, n1);
            for (int e = tid; e < (ev - skip) * VPR; e += nth) {
                const int x = skip + e / VPR, v8 = e % VPR, row = emap[x];
                const int slotc = (ch0 + cn0 + x) % a.C;
                const size_t off = ((size_t)u * a.C + slotc) * D;
                reinterpret_cast<uint4 *>(a.ck + off)[v8] = reinterpret_cast<const uint4 *>(ck + (size_t)row * RS)[RL::chunk(row, v8)];
                reinterpret_cast<uint4 *>(a.cv + off)[v8] = reinterpret_cast<const uint4 *>(cv + (size_t)row * RS)[RL::chunk(row, v8)];
                if (v8 == 0) a.cidx[(size_t)u * a.C + slotc] = (int32_t)(uint32_t)key[row];
            }
            if (tid == 0) {
                a.cmeta[2 * u] = n1;
                a.cmeta[2 * u + 1] = (ch0 + cn0 + ev - n1) % a.C;
            }
        }
    }

    // the block's slot: its own, or (paged pool) one taken from the free
    // slots; the host has checked that enough are free
    size_t slot = (size_t)u * a.NB + jj;
    if (a.bt) {
        if (tid == 0) {
            const int top = atomicSub(a.ftop, 1) - 1;
            if (top >= 0) {
                a.bt[slot] = a.fstack[top];
            } else {   // never with the host's count; recorded instead of reading out of bounds
                a.bt[slot] = 0;
                atomicExch(a.ctl + 1, 1);
            }
        }
        __syncthreads();
        slot = (size_t)__ldcg(a.bt + slot);
    }
    uint8_t *bb = a.blk + slot * a.blk_bytes;
    uint8_t *tiles = bb + ksz_bytes(D);
    for (int t = tid; t < G; t += nth)
        a.bidx[((size_t)u * a.NB + jj) * G + t] = t < cnt ? (int32_t)(uint32_t)key[bmap[t]] : -1;

    // 6. keys: one (scale, zero) per channel over the block's tokens. Each
    // thread takes a channel pair over one slice of the tokens (min/max of
    // ordered keys, two channels per SIMD instruction); the slices combine.
    {
        constexpr int NCP = D / 2;
        const int nsl = nth / NCP;
        uint32_t *kpart = reinterpret_cast<uint32_t *>(vrule);   // [nsl][2][D/2] key pairs
        const int cp = tid % NCP, sl = tid / NCP;
        const int tb = (cnt * sl) / nsl, te = (cnt * (sl + 1)) / nsl;
        uint32_t mn = 0x7fff7fffu, mx = 0x80008000u;
        for (int t = tb; t < te; ++t) {
            const int rw = bmap[t];
            const uint32_t k2 = okey2(*reinterpret_cast<const uint32_t *>(ck + (size_t)rw * RS + RL::pos(rw, 2 * cp)));
            mn = __vmins2(mn, k2);
            mx = __vmaxs2(mx, k2);
        }
        kpart[(size_t)sl * D + cp] = mn;
        kpart[(size_t)sl * D + NCP + cp] = mx;
        __syncthreads();
        for (int c2 = tid; c2 < NCP; c2 += nth) {
            uint32_t m0 = kpart[c2], m1 = kpart[NCP + c2];
            for (int q = 1; q < nsl; ++q) {
                m0 = __vmins2(m0, kpart[(size_t)q * D + c2]);
                m1 = __vmaxs2(m1, kpart[(size_t)q * D + NCP + c2]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int ch = 2 * c2 + h;
                __half s16 = __ushort_as_half(0), z16 = __ushort_as_half(0);
                if (cnt > 0) {
                    const float lo = okey_lo(m0 >> (16 * h)), hi = okey_lo(m1 >> (16 * h));
                    s16 = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 3.0f));
                    z16 = __float2half_rn(lo);
                }
                reinterpret_cast<uint32_t *>(bb)[ch] = half2_bits(s16, z16);
                krule[ch + (ch >> 3)] = code_rule(__half2float(s16), __half2float(z16));
            }
        }
        __syncthreads();   // the partials are read before the value rules overwrite them
    }
    // 7. values: one (scale, zero) per token per 32 channels (consecutive
    // threads take consecutive tokens of one group)
    for (int e = tid; e < TS * NG; e += nth) {
        const int t = e % TS, gm = e / TS;
        __half s16 = __ushort_as_half(0), z16 = __ushort_as_half(0);
        if (t < cnt) {
            const int rw = bmap[t];
            const uint4 *row = reinterpret_cast<const uint4 *>(cv + (size_t)rw * RS);
            uint32_t m0 = 0x7fff7fffu, m1 = 0x80008000u;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 x = row[RL::chunk(rw, 4 * gm + k)];
                const uint32_t w4[4] = {okey2(x.x), okey2(x.y), okey2(x.z), okey2(x.w)};
#pragma unroll
                for (int e2 = 0; e2 < 4; ++e2) {
                    m0 = __vmins2(m0, w4[e2]);
                    m1 = __vmaxs2(m1, w4[e2]);
                }
            }
            m0 = __vmins2(m0, m0 >> 16);   // the low lane takes the smaller of the two
            m1 = __vmaxs2(m1, __byte_perm(m1, 0, 0x3232));
            const float mn = okey_lo(m0), mx = okey_lo(m1);
            s16 = __float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f));
            z16 = __float2half_rn(mn);
            vrule[gm * VS + t + (t >> 3)] = code_rule(__half2float(s16), __half2float(z16));
        }
        uint8_t *tb = tiles + (size_t)(t / TILE) * tile_bytes(D) + tile_sz_off(D);
        reinterpret_cast<uint32_t *>(tb)[vsz_index(t, gm)] = half2_bits(s16, z16);
    }
    __syncthreads();

    // 8. pack the codes into the mma.sync word format (see ott_internal.cuh)
    const int nwords = a.ntile * 32 * NW;
    for (int e = tid; e < nwords; e += nth) {
        const int tau = e / (32 * NW), rem = e % (32 * NW), ln = rem / NW, w = rem % NW;
        const int r = ln >> 2, i = ln & 3, wp = w >> 1, hi = w & 1;
        uint32_t kw = 0, vw = 0;
        const int tk = TILE * tau + r + 8 * hi;   // K: token slot of this word
        if (tk < cnt) {
            const int rk_ = bmap[tk];
            const __half *krow = ck + (size_t)rk_ * RS;
#pragma unroll
            for (int p = 0; p < 8; ++p) {
                // K word: channels 16kt + 2i + 8o (+1) of token tk
                const int q = 8 * wp + p, o = q / NKT, kt = q % NKT, ch = 16 * kt + 2 * i + 8 * o;
                const uint32_t x2 = *reinterpret_cast<const uint32_t *>(krow + RL::pos(rk_, ch));
                const float4 r0 = krule[ch + (ch >> 3)], r1 = krule[ch + 1 + ((ch + 1) >> 3)];
                kw |= qcode_a(sub_h(x2, false, r0.x), r0) << (2 * p);
                kw |= qcode_a(sub_h(x2, true, r1.x), r1) << (16 + 2 * p);
            }
        }
        // V word: channel 16mt + r + 8rowhalf of token slots 16tau + 2i + 8hi (+1)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int tv = TILE * tau + 2 * i + 8 * hi + h;
            if (tv < cnt) {
                const int rv_ = bmap[tv];
                const __half *vrow = cv + (size_t)rv_ * RS;
                const float4 *vr = vrule + tv + (tv >> 3);
#pragma unroll
                for (int p = 0; p < 8; ++p) {
                    const int q = 8 * wp + p, rowhalf = q / NKT, mt = q % NKT, vch = 16 * mt + r + 8 * rowhalf;
                    const float4 rr = vr[(vch / 32) * VS];
                    const uint32_t x1 = __half_as_ushort(vrow[RL::pos(rv_, vch)]);
                    vw |= qcode_a(sub_h(x1, false, rr.x), rr) << (16 * h + 2 * p);
                }
            }
        }
        uint8_t *tb = tiles + (size_t)tau * tile_bytes(D);
        reinterpret_cast<uint32_t *>(tb + tile_k_off(D))[ln * NW + w] = kw;
        reinterpret_cast<uint32_t *>(tb + tile_v_off(D))[ln * NW + w] = vw;
    }
}

// Parallel prefill. The pool after flush j is the min(P, (j + 1) G) smallest
// (norm, index) keys among every token flushed so far (keeping the smallest
// of a union is associative), so it can be found for all j before any block
// is built, and then every flush of the prefill runs at once: pass 1 finds
// each group's own smallest keys, pass 2 merges them unit by unit into the
// pool history, pass 3 (k_flush with the history) builds every block.
constexpr int PF_THREADS = 128;
// shared memory of k_pf_group: G staged key rows of d + 8 halves, G keys
inline size_t pf_group_smem_bytes(int d, int G) { return (size_t)G * (d + 8) * 2 + (size_t)G * 8; }

// Pass 1, one CTA per group j of unit u0 + i: the G keys' squared norms,
// summed in fp32 in channel order exactly as k_flush sums them, and the
// group's min(P, G) smallest keys, ascending (no other group token can be in
// the pool after this group's flush).
template <int D>
__global__ void __launch_bounds__(PF_THREADS) k_pf_group(const __half *__restrict__ srcK, long long src_unit_stride,
                                                         int src_u0, int u0, int nf, int G, int P,
                                                         uint64_t *__restrict__ gtop) {
    // the group's keys, staged by coalesced asynchronous copies into rows
    // padded to D + 8 halves (each thread then reads its own row without
    // bank conflicts), and the group's (norm, index) keys
    constexpr int RS = D + 8, VPR = D / 8;
    extern __shared__ __align__(16) uint8_t pf_sm[];
    __half *rows = reinterpret_cast<__half *>(pf_sm);
    uint64_t *gkey = reinterpret_cast<uint64_t *>(pf_sm + (size_t)G * RS * 2);   // [G]
    const int uu = blockIdx.x / nf, j = blockIdx.x % nf, u = u0 + uu;
    const long long t0 = (long long)j * G;
    const __half *base = srcK + (size_t)(u - src_u0) * src_unit_stride + (size_t)t0 * D;
    for (int e = threadIdx.x; e < G * VPR; e += blockDim.x) {
        const int r = e / VPR, v8 = e % VPR;
        cp_async16(rows + (size_t)r * RS + 8 * v8, base + (size_t)r * D + 8 * v8);
    }
    cp_async_wait_all();
    __syncthreads();
    for (int t = threadIdx.x; t < G; t += blockDim.x) {
        const uint4 *row = reinterpret_cast<const uint4 *>(rows + (size_t)t * RS);
        float s = 0.0f;
#pragma unroll 4
        for (int v8 = 0; v8 < VPR; ++v8) {
            const uint4 x = row[v8];
            const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {   // channels 8 v8 + 2e, 8 v8 + 2e + 1
                s = sq_acc(w4[e], false, s);
                s = sq_acc(w4[e], true, s);
            }
        }
        gkey[t] = ((uint64_t)__float_as_uint(s) << 32) | (uint32_t)(t0 + t);
    }
    __syncthreads();
    const int nb = min(P, G);
    uint64_t *dst = gtop + ((size_t)uu * nf + j) * P;
    for (int t = threadIdx.x; t < G; t += blockDim.x) {
        const uint64_t k = gkey[t];
        int r = 0;
        for (int q = 0; q < G; ++q) r += gkey[q] < k;
        if (r < nb) dst[r] = k;
    }
}


// Outputs [k0, k1) (0-based, k1 <= na + nb) of the merge of the ascending
// lists A (na keys) and B (nb keys), all keys distinct, through emit(k, key):
// a binary search on the merge path finds how many of A's keys precede
// output k0, then each output takes the smaller head.
template <typename Emit>
__device__ __forceinline__ void merge_range(const uint64_t *A, int na, const uint64_t *B, int nb, int k0, int k1,
                                            Emit emit) {
    if (k0 >= k1) return;
    int ia = 0;   // A's keys among the first k0 outputs
    if (k0 > 0) {
        int lo = max(0, k0 - nb), hi = min(k0, na);
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (A[mid] < B[k0 - 1 - mid]) lo = mid + 1;
            else hi = mid;
        }
        ia = lo;
    }
    for (int k = k0; k < k1; ++k) {
        const int ib = k - ia;
        if (ia < na && (ib >= nb || A[ia] < B[ib])) emit(k, A[ia++]);
        else emit(k, B[ib]);
    }
}
// this lane's share of m outputs: a contiguous range
__device__ __forceinline__ void lane_range(int m, int lane, int &k0, int &k1) {
    const int per = (m + 31) >> 5;
    k0 = min(m, lane * per);
    k1 = min(m, k0 + per);
}

// Pass 2: the pool after flush j (ascending keys) is the smallest
// min(P, (j + 1) G) of groups 0..j's smallest keys. Keeping the smallest of
// a union is associative, so the pools are found by a scan. A unit's groups
// are cut into C chunks of cg groups, one CTA each (C > 1 when few units
// would leave SMs idle), and each CTA scans its chunk in two levels:
//   1. warp w scans its own range of the chunk's groups [j0, j1) alone: the
//      local prefix after group j (the smallest of groups j0..j), written to
//      the history;
//   2. the warps' totals are scanned across the warps (log2(warps) rounds of
//      merges, all warps at once): warp w's carry is the smallest of the
//      chunk's groups before j0;
//   3. warp w merges its carry into each of its local prefixes.
// The dependent merges per chunk are about 2 cg / warps + log2(warps). With
// C > 1 each CTA leaves its chunk's total in gtot, and k_pf_carry then merges
// the totals of the chunks before each chunk into that chunk's prefixes.
// Each lane takes a contiguous range of a merge's outputs (merge_range). The
// lists a warp merges next arrive by cp.async, SCAN_AHEAD of them in flight.
constexpr int SCAN_WARPS = 32;
constexpr int SCAN_AHEAD = 4;

// Shared memory of k_pf_scan for sw warps: per warp the running list, its
// successor and SCAN_AHEAD incoming lists; two lists per warp for the scan of
// the chunk totals, and their lengths.
inline size_t scan_smem_bytes(int sw, int P) {
    return (size_t)sw * P * (2 + SCAN_AHEAD + 2) * 8 + (size_t)sw * 2 * 4;
}

__global__ void __launch_bounds__(SCAN_WARPS * 32) k_pf_scan(const uint64_t *__restrict__ gtop,
                                                             uint64_t *__restrict__ phist, int nf_unit, int G, int P,
                                                             int cg, int C, uint64_t *__restrict__ gtot) {
    extern __shared__ uint64_t scan_sm[];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int uu = blockIdx.x / C, cc = blockIdx.x % C;
    uint64_t *A = scan_sm + (size_t)w * (2 + SCAN_AHEAD) * P, *Cn = A + P, *ring = Cn + P;
    uint64_t *Sa = scan_sm + (size_t)nw * (2 + SCAN_AHEAD) * P, *Sb = Sa + (size_t)nw * P;
    int *na_ = reinterpret_cast<int *>(Sb + (size_t)nw * P), *nb_ = na_ + nw;
    const int nb = min(P, G);
    // this CTA's chunk: groups [J0, J0 + nf) of the unit, scanned as if alone
    const int J0 = cc * cg, nf = min(nf_unit - J0, cg);
    const uint64_t *gt = gtop + ((size_t)uu * nf_unit + J0) * P;
    uint64_t *ph = phist + ((size_t)uu * nf_unit + J0) * P;
    // a warp's range may be empty (a short last chunk)
    const int j0 = (int)((long long)nf * w / nw), j1 = (int)((long long)nf * (w + 1) / nw);
    // list q of the ring <- n keys from src; always one commit group (possibly
    // empty), so that the list of step j is the one SCAN_AHEAD - 1 commits back
    auto fetch = [&](int q, const uint64_t *src, int n) {
        for (int k = lane; k < n; k += 32) cp_async8(ring + (size_t)q * P + k, src + k);
        cp_async_commit();
    };
    // 1. local prefixes of this warp's range
    for (int q = 0; q < SCAN_AHEAD; ++q) fetch(q, gt + (size_t)(j0 + q) * P, j0 + q < j1 ? nb : 0);
    int na = 0;
    for (int j = j0; j < j1; ++j) {
        const int q = (j - j0) % SCAN_AHEAD;
        cp_async_wait_group<SCAN_AHEAD - 1>();
        __syncwarp();
        const uint64_t *Bc = ring + (size_t)q * P;
        const int m = (int)min((long long)P, (long long)na + G);
        int k0, k1;
        lane_range(m, lane, k0, k1);
        merge_range(A, na, Bc, nb, k0, k1, [&](int k, uint64_t x) {
            Cn[k] = x;
            ph[(size_t)j * P + k] = x;
        });
        __syncwarp();
        fetch(q, gt + (size_t)(j + SCAN_AHEAD) * P, j + SCAN_AHEAD < j1 ? nb : 0);
        uint64_t *t = A; A = Cn; Cn = t;
        na = m;
    }
    for (int k = lane; k < na; k += 32) Sa[(size_t)w * P + k] = A[k];
    if (lane == 0) na_[w] = na;
    __syncthreads();
    // 2. inclusive scan of the warps' totals (Hillis-Steele): after it Sa[w]
    // is the smallest of warp ranges 0..w
    for (int dd = 1; dd < nw; dd <<= 1) {
        const uint64_t *x = Sa + (size_t)w * P;
        uint64_t *y = Sb + (size_t)w * P;
        if (w >= dd) {
            const int nx = na_[w - dd], ny = na_[w], m = min(P, nx + ny);
            int k0, k1;
            lane_range(m, lane, k0, k1);
            merge_range(Sa + (size_t)(w - dd) * P, nx, x, ny, k0, k1, [&](int k, uint64_t v) { y[k] = v; });
            if (lane == 0) nb_[w] = m;
        } else {
            for (int k = lane; k < na_[w]; k += 32) y[k] = x[k];
            if (lane == 0) nb_[w] = na_[w];
        }
        __syncthreads();
        uint64_t *t = Sa; Sa = Sb; Sb = t;
        int *ti = na_; na_ = nb_; nb_ = ti;
    }
    // the chunk's total (the smallest of all its groups) for the carries
    if (C > 1 && w == nw - 1) {
        uint64_t *dst = gtot + ((size_t)uu * C + cc) * P;
        for (int k = lane; k < na_[nw - 1]; k += 32) dst[k] = Sa[(size_t)(nw - 1) * P + k];
    }
    // 3. the pool after group j: the carry (the warp ranges before this one)
    // merged with the local prefix
    if (w > 0) {
        const uint64_t *cw = Sa + (size_t)(w - 1) * P;
        const int ncar = na_[w - 1];
        auto nl_of = [&](int j) { return (int)min((long long)P, (long long)(j - j0 + 1) * G); };
        for (int q = 0; q < SCAN_AHEAD; ++q) fetch(q, ph + (size_t)(j0 + q) * P, j0 + q < j1 ? nl_of(j0 + q) : 0);
        for (int j = j0; j < j1; ++j) {
            const int q = (j - j0) % SCAN_AHEAD;
            cp_async_wait_group<SCAN_AHEAD - 1>();
            __syncwarp();
            const int nl = nl_of(j), m = (int)min((long long)P, (long long)(j + 1) * G);
            int k0, k1;
            lane_range(m, lane, k0, k1);
            merge_range(cw, ncar, ring + (size_t)q * P, nl, k0, k1, [&](int k, uint64_t v) { ph[(size_t)j * P + k] = v; });
            __syncwarp();
            fetch(q, ph + (size_t)(j + SCAN_AHEAD) * P, j + SCAN_AHEAD < j1 ? nl_of(j + SCAN_AHEAD) : 0);
        }
    }
    cp_async_wait_group<0>();
}

// Pass 2b (C > 1), one CTA per unit and chunk c >= 1: the carry of chunk c,
// the smallest of chunks 0..c-1 (their totals reduced pairwise in
// ceil(log2 c) rounds), merged into each of its groups' prefixes.
constexpr int CARRY_MAX_CHUNKS = 32;

inline size_t carry_smem_bytes(int C, int nw, int P) { return ((size_t)2 * C + nw) * P * 8; }

__global__ void __launch_bounds__(SCAN_WARPS * 32) k_pf_carry(uint64_t *__restrict__ phist,
                                                              const uint64_t *__restrict__ gtot, int nf, int G,
                                                              int P, int cg, int C) {
    extern __shared__ uint64_t car_sm[];
    __shared__ int cnt[2][CARRY_MAX_CHUNKS];
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int uu = blockIdx.x / (C - 1), c = blockIdx.x % (C - 1) + 1;
    uint64_t *La = car_sm, *Lb = car_sm + (size_t)C * P, *Bw = car_sm + (size_t)2 * C * P + (size_t)w * P;
    int *ca = cnt[0], *cb = cnt[1];
    // the totals of chunks 0..c-1 (chunk x holds min(P, its groups x G) keys)
    for (int x = threadIdx.x; x < c; x += blockDim.x)
        ca[x] = (int)min((long long)P, (long long)min(cg, nf - x * cg) * G);
    __syncthreads();
    for (int e = threadIdx.x; e < c * P; e += blockDim.x) {
        const int x = e / P, k = e % P;
        if (k < ca[x]) La[e] = gtot[((size_t)uu * C + x) * P + k];
    }
    __syncthreads();
    for (int n = c; n > 1;) {
        const int half = (n + 1) / 2;
        for (int pi = w; pi < half; pi += nw) {
            const int x = 2 * pi;
            uint64_t *y = Lb + (size_t)pi * P;
            if (x + 1 < n) {
                const int m = min(P, ca[x] + ca[x + 1]);
                int k0, k1;
                lane_range(m, lane, k0, k1);
                merge_range(La + (size_t)x * P, ca[x], La + (size_t)(x + 1) * P, ca[x + 1], k0, k1,
                            [&](int k, uint64_t v) { y[k] = v; });
                if (lane == 0) cb[pi] = m;
            } else {
                for (int k = lane; k < ca[x]; k += 32) y[k] = La[(size_t)x * P + k];
                if (lane == 0) cb[pi] = ca[x];
            }
        }
        __syncthreads();
        uint64_t *t = La; La = Lb; Lb = t;
        int *ti = ca; ca = cb; cb = ti;
        n = half;
    }
    const int ncar = ca[0];
    const int J0 = c * cg, J1 = min(nf, J0 + cg);
    for (int j = J0 + w; j < J1; j += nw) {
        const int nl = (int)min((long long)P, (long long)(j - J0 + 1) * G), m = (int)min((long long)P, (long long)(j + 1) * G);
        uint64_t *pj = phist + ((size_t)uu * nf + j) * P;
        for (int k = lane; k < nl; k += 32) Bw[k] = pj[k];
        __syncwarp();
        int k0, k1;
        lane_range(m, lane, k0, k1);
        merge_range(La, ncar, Bw, nl, k0, k1, [&](int k, uint64_t v) { pj[k] = v; });
        __syncwarp();
    }
}

// k, v [U][d] -> ring slot `slot` of every unit
// With qsrc, the step's queries (nq 16-byte vectors) are copied to qdst too
// (a step fed from host memory: k, v and q are read where they are).
__global__ void k_append(const uint4 *__restrict__ k, const uint4 *__restrict__ v, __half *rk,
                         __half *rv, int U, int d, int ring, int slot, const uint4 *__restrict__ qsrc,
                         uint4 *__restrict__ qdst, int nq) {
    // a decode queued next may start now; it waits for this grid before reading the ring
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // launched as a programmatic dependent: the kernel before this one (the
    // previous call's combine, or whatever wrote k and v) completes first
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // one 16-byte vector per thread (k and v of one unit, or one of q), so
    // that every load is in flight at once (they may come from host memory)
    const int vpr = d / 8, n = U * vpr;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n + nq; e += gridDim.x * blockDim.x) {
        if (e < n) {
            const int u = e / vpr, x = e % vpr;
            const size_t off = ((size_t)u * ring + slot) * d;
            const uint4 kk = k[e], vv = v[e];
            reinterpret_cast<uint4 *>(rk + off)[x] = kk;
            reinterpret_cast<uint4 *>(rv + off)[x] = vv;
        } else {
            qdst[e - n] = qsrc[e - n];
        }
    }
}

// Ragged batches: k, v [U][d] -> ring slot slot[b] of every unit of sequence b.
struct SlotTable {
    int slot[RAGGED_MAX];
};

__global__ void k_append_ragged(const uint4 *__restrict__ k, const uint4 *__restrict__ v, __half *rk,
                                __half *rv, int U, int Hkv, int d, int ring, const __grid_constant__ SlotTable st,
                                const uint4 *__restrict__ qsrc, uint4 *__restrict__ qdst, int nq) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int vpr = d / 8, n = U * vpr;
    for (int e = blockIdx.x * blockDim.x + threadIdx.x; e < n + nq; e += gridDim.x * blockDim.x) {
        if (e < n) {
            const int u = e / vpr, x = e % vpr;
            const size_t off = ((size_t)u * ring + st.slot[u / Hkv]) * d;
            const uint4 kk = k[e], vv = v[e];
            reinterpret_cast<uint4 *>(rk + off)[x] = kk;
            reinterpret_cast<uint4 *>(rv + off)[x] = vv;
        } else {
            qdst[e - n] = qsrc[e - n];
        }
    }
}

// tokens [t_begin, t_end) of units [u0, u0+nu) of K, V [U][Lstride][d] -> their ring slots
__global__ void k_copy_tail(const __half *K, const __half *V, __half *rk, __half *rv, int u0, int nu, int d,
                            int ring, int Lstride, long long t_begin, long long t_end, int src_u0) {
    const int vpr = d / 8;
    const long long ntok = t_end - t_begin;
    const long long total = (long long)nu * ntok * vpr;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const int x = (int)(e % vpr);
        const long long tt = (e / vpr) % ntok;
        const int u = u0 + (int)(e / vpr / ntok);
        const long long t = t_begin + tt;
        const size_t src = ((size_t)(u - src_u0) * Lstride + t) * d;
        const size_t dst = ((size_t)u * ring + (size_t)(t % ring)) * d;
        reinterpret_cast<uint4 *>(rk + dst)[x] = reinterpret_cast<const uint4 *>(K + src)[x];
        reinterpret_cast<uint4 *>(rv + dst)[x] = reinterpret_cast<const uint4 *>(V + src)[x];
    }
}

// Canonical export of the quantized blocks of units [u0, u0+nu):
//   kcode/vcode [nu][nf][G][d/4] bytes, ks/kz [nu][nf][d], vs/vz [nu][nf][G][d/32]
struct ExportArgs {
    const uint8_t *blk;
    const int32_t *bt;       // paged pool: slot of each block (null: u*NB + j)
    long long blk_bytes;
    int NB, nf, G, d, u0, nu;
    uint8_t *kcode, *vcode;
    uint16_t *ks, *kz, *vs, *vz;
};

__device__ __forceinline__ size_t export_slot(const ExportArgs &a, int u, int j) {
    const size_t own = (size_t)u * a.NB + j;
    return a.bt ? (size_t)a.bt[own] : own;
}

__global__ void k_export(ExportArgs a) {
    const int d = a.d, rb = d / 4, NG = d / 32;
    const long long nblk = (long long)a.nu * a.nf;
    const long long n_code = nblk * a.G * rb;
    const long long n_ksz = nblk * d;
    const long long n_vsz = nblk * a.G * NG;
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n_code; e += stride) {
        const int by = (int)(e % rb);
        const int t = (int)((e / rb) % a.G);
        const long long bj = e / rb / a.G;
        const int j = (int)(bj % a.nf), uu = (int)(bj / a.nf);
        const uint8_t *tb = a.blk + export_slot(a, a.u0 + uu, j) * a.blk_bytes + ksz_bytes(d) +
                            (size_t)(t / TILE) * tile_bytes(d);
        const uint32_t *kw = reinterpret_cast<const uint32_t *>(tb + tile_k_off(d));
        const uint32_t *vw = reinterpret_cast<const uint32_t *>(tb + tile_v_off(d));
        uint32_t kb = 0, vb = 0;
        for (int x = 0; x < 4; ++x) {
            const int ch = 4 * by + x;
            int w, bit;
            k_loc(t, ch, d, w, bit);
            kb |= ((kw[w] >> bit) & 3u) << (2 * x);
            v_loc(t, ch, d, w, bit);
            vb |= ((vw[w] >> bit) & 3u) << (2 * x);
        }
        a.kcode[e] = (uint8_t)kb;
        a.vcode[e] = (uint8_t)vb;
    }
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n_ksz; e += stride) {
        const int ch = (int)(e % d);
        const long long bj = e / d;
        const int j = (int)(bj % a.nf), uu = (int)(bj / a.nf);
        const uint32_t sz = reinterpret_cast<const uint32_t *>(a.blk + export_slot(a, a.u0 + uu, j) * a.blk_bytes)[ch];
        a.ks[e] = (uint16_t)(sz & 0xffffu);
        a.kz[e] = (uint16_t)(sz >> 16);
    }
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n_vsz; e += stride) {
        const int gm = (int)(e % NG);
        const int t = (int)((e / NG) % a.G);
        const long long bj = e / NG / a.G;
        const int j = (int)(bj % a.nf), uu = (int)(bj / a.nf);
        const uint8_t *tb = a.blk + export_slot(a, a.u0 + uu, j) * a.blk_bytes + ksz_bytes(d) +
                            (size_t)(t / TILE) * tile_bytes(d);
        const uint32_t sz = reinterpret_cast<const uint32_t *>(tb + tile_sz_off(d))[vsz_index(t, gm)];
        a.vs[e] = (uint16_t)(sz & 0xffffu);
        a.vz[e] = (uint16_t)(sz >> 16);
    }
}

}  // namespace

namespace {

long long flush_smem_layout(int d, int G, int P, bool sw) {
    const long long nc = (long long)P + G;
    const long long b = nc * (sw ? d : d + 8) * 2 * 2   // staged K and V rows
                        + nc * 8               // keys
                        + nc * 4 + (long long)G * 4           // ranks, block map
                        + (long long)(P > 0 ? P : 1) * 4      // cold order
                        + 16                                  // alignment of the code rules
                        + (long long)(d + d / 8) * 16;        // key code rules (skewed)
    // value code rules (skewed), an area that first holds the key min/max partials
    const long long ts = (long long)ntiles_of(G) * TILE;
    const long long vr = (ts + ts / 8) * (d / 32) * 16;
    const long long kp = (long long)(FLUSH_THREADS / (d / 2)) * 2 * d * 4;
    return b + (vr > kp ? vr : kp);
}

// Swizzled rows only where they let a second CTA share the SM (its 228 KB of
// shared memory, 1 KB reserved per CTA) and padded rows would not: the
// swizzle costs address arithmetic in an issue-bound kernel.
bool flush_swizzle(int d, int G, int P) {
    constexpr long long SM_SMEM = 228 * 1024, RESERVED = 1024;
    const bool two_padded = 2 * (flush_smem_layout(d, G, P, false) + RESERVED) <= SM_SMEM;
    const bool two_swizzled = 2 * (flush_smem_layout(d, G, P, true) + RESERVED) <= SM_SMEM;
    return !two_padded && two_swizzled;
}

bool flush_swizzled(const ott_cache *c) { return flush_swizzle(c->d, c->G, c->P); }

}  // namespace

int flush_smem_bytes(int d, int G, int P) {
    const long long t = flush_smem_layout(d, G, P, flush_swizzle(d, G, P));
    return t > (1LL << 30) ? (1 << 30) : (int)t;
}

namespace {

// An append is launched as a programmatic dependent of the kernel before it:
// it releases its own dependents at once and then waits for that kernel, so
// only its launch overlaps the previous kernel's tail.
cudaLaunchConfig_t pdl_config(int blocks, int threads, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    return cfg;
}

void pdl_attr(cudaLaunchConfig_t &cfg, cudaLaunchAttribute (&attr)[1]) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
}

}  // namespace

cudaError_t launch_append(const ott_cache *c, const __half *k, const __half *v, cudaStream_t s, const __half *qsrc) {
    const int slot = (int)(c->T % c->ring);
    const int n = c->U * c->d / 8;
    const int nq = qsrc ? c->B * c->Hq * c->d / 8 : 0;
    const int th = 256, bl = (n + nq + th - 1) / th;
    cudaLaunchConfig_t cfg = pdl_config(bl, th, s);
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, k_append, reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v),
                              c->rk, c->rv, c->U, c->d, c->ring, slot, reinterpret_cast<const uint4 *>(qsrc),
                              reinterpret_cast<uint4 *>(c->qdev), nq);
}

namespace {

FlushArgs flush_args(const ott_cache *c, const __half *srcK, const __half *srcV, long long src_unit_stride,
                     long long src_mod, long long t0, int j) {
    FlushArgs a;
    a.blk = c->blk;
    a.bidx = c->bidx;
    a.pk = c->pk;
    a.pv = c->pv;
    a.pnorm = c->pnorm;
    a.pidx = c->pidx;
    a.srcK = srcK;
    a.srcV = srcV;
    a.ck = c->ck;
    a.cv = c->cv;
    a.cidx = c->cidx;
    a.cmeta = c->cmeta;
    a.bcnt = c->bcnt;
    a.C = c->cold;
    a.bt = c->paged ? c->bt : nullptr;
    a.fstack = c->fstack;
    a.ftop = c->ftop;
    a.ctl = c->ctl;
    a.src_u0 = 0;
    a.phist = nullptr;
    a.pf_nf = 0;
    a.pf_u0 = 0;
    a.src_unit_stride = src_unit_stride;
    a.src_mod = src_mod;
    a.t0 = t0;
    a.blk_bytes = c->blk_bytes;
    a.G = c->G;
    a.P = c->P;
    a.NB = c->NB;
    a.ntile = c->ntile;
    a.j = j;
    a.np0 = pool_after(c->P, c->G, j, c->pct);
    a.pct = c->pct;
    a.n_oc = c->n_oc;
    a.Hkv = c->Hkv;
    return a;
}

cudaError_t run_flush(const ott_cache *c, const FlushArgs &a, const FlushList &fl, int ctas, cudaStream_t s) {
    const int smem = flush_smem_bytes(c->d, c->G, c->P);
    if (c->d == 128)
        flush_swizzled(c) ? k_flush<128, true><<<ctas, FLUSH_THREADS, smem, s>>>(a, fl)
                          : k_flush<128, false><<<ctas, FLUSH_THREADS, smem, s>>>(a, fl);
    else
        flush_swizzled(c) ? k_flush<64, true><<<ctas, FLUSH_THREADS, smem, s>>>(a, fl)
                          : k_flush<64, false><<<ctas, FLUSH_THREADS, smem, s>>>(a, fl);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_flush(const ott_cache *c, const __half *srcK, const __half *srcV,
                         long long src_unit_stride, long long src_mod, long long t0, int j,
                         cudaStream_t s) {
    FlushList none;
    none.n = 0;
    return run_flush(c, flush_args(c, srcK, srcV, src_unit_stride, src_mod, t0, j), none, c->U, s);
}

bool prefill_parallel_ok(const ott_cache *c, int nf, int shared_units) {
    // The cold pool and the channel criterion carry state that a flush needs
    // from the one before it. A call that covers all its units in one pass
    // (shared_units = 0) always takes it: its one launch of every block has
    // no idle tails and no sequential launches (measured, 4,096-token
    // prompts: 1,024 units 1.72 ms against 1.76 ms group by group, 512 units
    // 0.89 against 1.05, 256 units 0.47 against 0.61). A ragged batch runs
    // one pass per sequence, one after another; there the group-by-group
    // launches, shared by every sequence, win once the shared_units they
    // carry fill the GPU.
    return c->cold < 0 && c->pct < 0 && nf >= 2 && shared_units < c->sm_count;
}

// Chunks per unit of the pool scan: enough CTAs to cover the SMs twice, at
// most CARRY_MAX_CHUNKS, and chunks of at least SCAN_WARPS groups.
static int scan_chunks(const ott_cache *c, int nu, int nf) {
    long long C = std::min<long long>(CARRY_MAX_CHUNKS, (nf + SCAN_WARPS - 1) / SCAN_WARPS);
    C = std::min<long long>(C, (2LL * c->sm_count + nu - 1) / nu);
    return C < 1 ? 1 : (int)C;
}

cudaError_t launch_prefill_parallel(const ott_cache *c, const __half *srcK, const __half *srcV,
                                    long long src_unit_stride, int src_u0, int u0, int nu, int nf,
                                    uint64_t *scratch, cudaStream_t s) {
    if (nu <= 0 || nf <= 0) return cudaSuccess;
    const int G = c->G, P = c->P;
    uint64_t *gtop = scratch, *phist = scratch + (size_t)nu * nf * P;
    const long long groups = (long long)nu * nf;
    if (groups > 0x7fffffffLL) return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    if (P > 0) {   // with no pool every block is its own group: pass 3 alone
    if (c->d == 128)
        k_pf_group<128><<<(int)groups, PF_THREADS, pf_group_smem_bytes(128, G), s>>>(
            srcK, src_unit_stride, src_u0, u0, nf, G, P, gtop);
    else
        k_pf_group<64><<<(int)groups, PF_THREADS, pf_group_smem_bytes(64, G), s>>>(
            srcK, src_unit_stride, src_u0, u0, nf, G, P, gtop);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // C chunks per unit, one CTA each; a warp per 4 groups of a chunk (fewer,
    // smaller CTAs cover the SMs in one wave), at most SCAN_WARPS, within
    // the shared memory
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    if (e != cudaSuccess) return e;
    const int C = scan_chunks(c, nu, nf), cg = (nf + C - 1) / C;
    uint64_t *gtot = C > 1 ? phist + (size_t)nu * nf * P : nullptr;
    int sw = (cg + 4 - 1) / 4;
    sw = sw < 1 ? 1 : (sw > SCAN_WARPS ? SCAN_WARPS : sw);
    while (sw > 1 && scan_smem_bytes(sw, P) > (size_t)optin) --sw;
    k_pf_scan<<<nu * C, 32 * sw, scan_smem_bytes(sw, P), s>>>(gtop, phist, nf, G, P, cg, C, gtot);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (C > 1) {
        int cw = cg < SCAN_WARPS ? cg : SCAN_WARPS;
        const size_t room = (size_t)optin - sizeof(int) * 2 * CARRY_MAX_CHUNKS;   // after the static counts
        while (cw > 1 && carry_smem_bytes(C, cw, P) > room) --cw;
        if (carry_smem_bytes(C, cw, P) > room) return cudaErrorInvalidValue;
        k_pf_carry<<<nu * (C - 1), 32 * cw, carry_smem_bytes(C, cw, P), s>>>(phist, gtot, nf, G, P, cg, C);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    }
    FlushArgs a = flush_args(c, srcK, srcV, src_unit_stride, LLONG_MAX, 0, 0);
    a.src_u0 = src_u0;
    a.phist = phist;
    a.pf_nf = nf;
    a.pf_u0 = u0;
    FlushList none;
    none.n = 0;
    return run_flush(c, a, none, (int)groups, s);
}

size_t prefill_scratch_bytes(const ott_cache *c, int nu, int nf) {
    const int C = scan_chunks(c, nu, nf);
    return (size_t)2 * nu * nf * c->P * 8 + (C > 1 ? (size_t)nu * C * c->P * 8 : 0) + 16;
}

cudaError_t launch_flush_list(const ott_cache *c, const __half *srcK, const __half *srcV,
                              long long src_unit_stride, long long src_mod, const FlushList &fl,
                              cudaStream_t s) {
    if (fl.n <= 0) return cudaSuccess;
    return run_flush(c, flush_args(c, srcK, srcV, src_unit_stride, src_mod, 0, 0), fl, fl.n * c->Hkv, s);
}

cudaError_t launch_flush_list_src(const ott_cache *c, const __half *srcK, const __half *srcV,
                                  long long src_unit_stride, long long src_mod, int src_u0, const FlushList &fl,
                                  cudaStream_t s) {
    if (fl.n <= 0) return cudaSuccess;
    FlushArgs a = flush_args(c, srcK, srcV, src_unit_stride, src_mod, 0, 0);
    a.src_u0 = src_u0;
    return run_flush(c, a, fl, fl.n * c->Hkv, s);
}

// Paged pool: the blocks of sequence b's units go back to the free slots.
__global__ void k_release(int32_t *fstack, int *ftop, const int32_t *bt, int u0, int NB, int nf, int pool,
                          int *ctl) {
    const int u = u0 + blockIdx.x;
    for (int j = threadIdx.x; j < nf; j += blockDim.x) {
        const int top = atomicAdd(ftop, 1);
        if (top < pool)
            fstack[top] = bt[(size_t)u * NB + j];
        else   // never with the host's count; recorded instead of writing out of bounds
            atomicExch(ctl + 1, 1);
    }
}

cudaError_t launch_release(const ott_cache *c, int b, cudaStream_t s) {
    const int nf = c->nfb[b];
    if (!c->paged || nf == 0) return cudaSuccess;
    k_release<<<c->Hkv, 256, 0, s>>>(c->fstack, c->ftop, c->bt, b * c->Hkv, c->NB, nf, c->pool_blocks, c->ctl);
    return cudaGetLastError();
}

cudaError_t launch_append_ragged(const ott_cache *c, const __half *k, const __half *v, cudaStream_t s,
                                 const __half *qsrc) {
    const int nq = qsrc ? c->B * c->Hq * c->d / 8 : 0;
    SlotTable st;
    for (int b = 0; b < c->B; ++b) st.slot[b] = (int)(c->Tb[b] % c->ring);
    const int n = c->U * c->d / 8;
    const int th = 256, bl = (n + nq + th - 1) / th;
    cudaLaunchConfig_t cfg = pdl_config(bl, th, s);
    cudaLaunchAttribute attr[1];
    pdl_attr(cfg, attr);
    return cudaLaunchKernelEx(&cfg, k_append_ragged, reinterpret_cast<const uint4 *>(k),
                              reinterpret_cast<const uint4 *>(v), c->rk, c->rv, c->U, c->Hkv, c->d, c->ring, st,
                              reinterpret_cast<const uint4 *>(qsrc), reinterpret_cast<uint4 *>(c->qdev), nq);
}

cudaError_t launch_copy_tail_units(const ott_cache *c, const __half *K, const __half *V, int u0, int nu,
                                   int Lstride, long long t_begin, long long t_end, cudaStream_t s, int src_u0) {
    if (t_begin >= t_end || nu <= 0) return cudaSuccess;
    const long long total = (long long)nu * (t_end - t_begin) * (c->d / 8);
    const int th = 256;
    const long long bl = (total + th - 1) / th;
    k_copy_tail<<<(int)(bl < 65535 ? bl : 65535), th, 0, s>>>(K, V, c->rk, c->rv, u0, nu, c->d, c->ring,
                                                               Lstride, t_begin, t_end, src_u0);
    return cudaGetLastError();
}

cudaError_t launch_copy_tail(const ott_cache *c, const __half *K, const __half *V, int L,
                             long long t_begin, cudaStream_t s) {
    return launch_copy_tail_units(c, K, V, 0, c->U, L, t_begin, L, s);
}

size_t export_stage_bytes(const ott_cache *c, int nu, int nf) {
    const size_t nblk = (size_t)nu * nf;
    return nblk * c->G * (c->d / 4) * 2 + nblk * c->d * 2 * 2 + nblk * c->G * (c->d / 32) * 2 * 2 + 64;
}

cudaError_t launch_export(const ott_cache *c, int u0, int nu, int nf, uint8_t *stage, cudaStream_t s) {
    const size_t nblk = (size_t)nu * nf;
    ExportArgs a;
    a.blk = c->blk;
    a.bt = c->paged ? c->bt : nullptr;
    a.blk_bytes = c->blk_bytes;
    a.NB = c->NB;
    a.nf = nf;
    a.G = c->G;
    a.d = c->d;
    a.u0 = u0;
    a.nu = nu;
    uint8_t *p = stage;
    a.kcode = p; p += nblk * c->G * (c->d / 4);
    a.vcode = p; p += nblk * c->G * (c->d / 4);
    a.ks = reinterpret_cast<uint16_t *>(p); p += nblk * c->d * 2;
    a.kz = reinterpret_cast<uint16_t *>(p); p += nblk * c->d * 2;
    a.vs = reinterpret_cast<uint16_t *>(p); p += nblk * c->G * (c->d / 32) * 2;
    a.vz = reinterpret_cast<uint16_t *>(p);
    if (nblk == 0) return cudaSuccess;
    k_export<<<4 * c->sm_count, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t set_flush_attributes(int d, int smem) {
    cudaError_t e = cudaFuncSetAttribute(k_pf_scan, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(k_pf_carry, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             smem - (int)sizeof(int) * 2 * CARRY_MAX_CHUNKS);
    if (e != cudaSuccess) return e;
    const void *fns[] = {reinterpret_cast<const void *>(k_flush<128, true>),
                         reinterpret_cast<const void *>(k_flush<128, false>),
                         reinterpret_cast<const void *>(k_flush<64, true>),
                         reinterpret_cast<const void *>(k_flush<64, false>),
                         reinterpret_cast<const void *>(k_pf_group<128>),
                         reinterpret_cast<const void *>(k_pf_group<64>)};
    for (const void *f : fns) {
        e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace ott
