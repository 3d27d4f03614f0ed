// ott_topk.cu -- block selection for Top-K sparse decode.
//
// "Accurate KV Cache Quantization with Outlier Tokens Tracing", zijie-tian.site
// sec. 6 names combining OTT with sparse access to the quantized KV as the
// next step. Here a decode call may attend only K quantized blocks of every
// (sequence, kv head), next to all residual and pool tokens: the non-empty
// blocks with the largest score bound, ties to the lower block index. The
// bound of block j for query head h is the largest q.k that a key
// dequantized from the block's per-channel scale s and zero z can reach,
// sum_c max(q_c z_c, q_c (z_c + 3 s_c)): each dequantized channel lies in
// [z_c, z_c + 3 s_c]. It is taken in fp32 with round-to-nearest products and
// sums in channel order, so that it is reproducible bit for bit; a block's
// bound is the largest over the query heads of its kv head.
//
// Two kernels, then the decode, chained by programmatic dependent launches
// (each starts while the previous one drains and waits for its results):
//   k_topk_bounds: a CTA of 128 threads per (unit, 32 blocks). The 32
//     blocks' K scale/zero headers (4d bytes each, the only part of a block
//     read here) are staged into shared memory, every thread with all its
//     16-byte loads in flight at once, in rows padded by one word so that the
//     threads of a warp, each reading one channel of its own block, hit
//     different banks. Thread (block, head) then sums its bound in channel
//     order; the block's bound is the largest over its heads.
//   k_topk_pick: a CTA per unit. An exact radix select over the bounds (four
//     8-bit histogram rounds) finds the first min(K, non-empty blocks) under
//     (bound descending, index ascending); a prefix count writes them to
//     sel[u][0..Kc) in ascending block order (-1 in the slots left over).
#include <math_constants.h>

#include "ott_internal.cuh"

namespace ott {
namespace {

constexpr int BND_BLOCKS = 32;      // blocks per bounds CTA
constexpr int BND_THREADS = 128;
constexpr int SORT_THREADS = 512;   // selection CTA: at most

struct TopkArgs {
    const uint8_t *blk;
    long long blk_bytes;
    int NB, nf, G, P, jfull;
    const int32_t *bcnt;     // block sizes under the cold-pool policy, else null
    const __half *q;         // [B][Hq][d]
    int Hq, Hkv;
    int g;                   // query heads per kv head (taken GQ at a time)
    int K;                   // blocks to keep
    int Kc;                  // slots per unit in sel: min(K, nf)
    float *bound;            // [U][NB] scratch: block bounds
    int32_t *sel;            // [U][Kc]
    const int32_t *bt;       // paged pool: slot of each block (null: u*NB + j)
    int ragged;              // 1: sequence b has nfb.nf[b] blocks (else nf for all)
};

// Blocks of each sequence of a ragged batch (a kernel parameter).
struct NfTable {
    int nf[RAGGED_MAX];
};

__device__ __forceinline__ int unit_nf(const TopkArgs &a, const NfTable &t, int u) {
    return a.ragged ? t.nf[u / a.Hkv] : a.nf;
}

template <int D, int GQ>
__global__ void __launch_bounds__(BND_THREADS) k_topk_bounds(TopkArgs a, const __grid_constant__ NfTable nt) {
    constexpr int RW = D + 1;                    // padded row (words)
    constexpr int V4 = D / 4;                    // 16-byte pieces per header
    constexpr int PER = BND_BLOCKS * V4 / BND_THREADS;
    static_assert(BND_BLOCKS * GQ <= BND_THREADS, "one thread per (block, head)");
    static_assert(BND_BLOCKS * V4 % BND_THREADS == 0, "whole pieces per thread");
    __shared__ uint32_t hdr[BND_BLOCKS * RW];
    __shared__ float qs[GQ * D];
    __shared__ float part[GQ][BND_BLOCKS];
    // the sort may be scheduled now; it waits for these bounds
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u = blockIdx.y, j0 = blockIdx.x * BND_BLOCKS, tid = threadIdx.x, nth = blockDim.x;
    const int nf_u = unit_nf(a, nt, u);
    if (j0 >= nf_u) return;   // the whole CTA: this unit has fewer blocks
    const int nb = min(BND_BLOCKS, nf_u - j0);
    const int b = u / a.Hkv, hk = u % a.Hkv;
    const __half *qp = a.q + ((size_t)b * a.Hq + (size_t)hk * a.g) * D;
    // the first GQ query heads (a kv head with fewer repeats its last one)
    auto load_q = [&](int s0) {
        for (int e = tid; e < GQ * D; e += nth) qs[e] = __half2float(qp[(size_t)min(s0 + e / D, a.g - 1) * D + e % D]);
    };
    load_q(0);
    uint4 buf[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = tid + i * BND_THREADS, r = e / V4, v = e % V4;
        if (r < nb) {
            const size_t own = (size_t)u * a.NB + j0 + r;
            const size_t slot = a.bt ? (size_t)__ldg(a.bt + own) : own;
            buf[i] = __ldg(reinterpret_cast<const uint4 *>(a.blk + slot * a.blk_bytes) + v);
        }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = tid + i * BND_THREADS, r = e / V4, v = e % V4;
        if (r < nb) {
            uint32_t *dst = hdr + r * RW + 4 * v;
            dst[0] = buf[i].x;
            dst[1] = buf[i].y;
            dst[2] = buf[i].z;
            dst[3] = buf[i].w;
        }
    }
    const int r = tid % BND_BLOCKS, h = tid / BND_BLOCKS;
    float best = -CUDART_INF_F;   // thread tid < nb: block j0 + tid, over the heads so far
    // the kv head's g query heads, GQ per round (a short last round repeats
    // its last head, which leaves the maximum unchanged)
    for (int s0 = 0; s0 < a.g; s0 += GQ) {
        if (s0 > 0) {
            __syncthreads();   // the previous round's heads and bounds are read
            load_q(s0);
        }
        __syncthreads();
        if (h < GQ && r < nb) {
            float acc = 0.0f;
            const uint32_t *row = hdr + r * RW;
            const float *qh = qs + h * D;
#pragma unroll 8
            for (int c = 0; c < D; ++c) {
                const uint32_t w = row[c];
                const float s = __half2float(__ushort_as_half((unsigned short)(w & 0xffffu)));
                const float z = __half2float(__ushort_as_half((unsigned short)(w >> 16)));
                const float top = __fadd_rn(z, __fmul_rn(3.0f, s));
                const float lo = __fmul_rn(qh[c], z), hi = __fmul_rn(qh[c], top);
                acc = __fadd_rn(acc, hi > lo ? hi : lo);
            }
            part[h][r] = acc;
        }
        __syncthreads();
        if (tid < nb)
#pragma unroll
            for (int x = 0; x < GQ; ++x) best = part[x][tid] > best ? part[x][tid] : best;
    }
    if (tid < nb) {
        const int j = j0 + tid;
        const int cnt = a.bcnt ? a.bcnt[(size_t)u * a.NB + j] : (j >= a.jfull ? a.G : block_count(a.P, a.G, j));
        a.bound[(size_t)u * a.NB + j] = cnt > 0 ? best : -CUDART_INF_F;
    }
}

// fp32 -> uint32 whose unsigned order is the float order
__device__ __forceinline__ uint32_t ordered(float f) {
    const uint32_t x = __float_as_uint(f);
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}

// Exclusive prefix sum of v over the threads of the CTA (in thread order);
// `total` receives the sum over all threads. ws: 32 ints of shared memory.
__device__ __forceinline__ int block_exscan(int v, int *ws, int &total) {
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) ws[wid] = x;
    __syncthreads();
    if (wid == 0) {
        int t = lane < nw ? ws[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, t, o);
            if (lane >= o) t += y;
        }
        ws[lane] = t;
    }
    __syncthreads();
    total = ws[nw - 1];
    const int r = (wid > 0 ? ws[wid - 1] : 0) + x - v;
    __syncthreads();   // ws is reused by the next call
    return r;
}

// The selection, by an exact radix select: key_j = the bit-inverted ordered
// bound (smallest key = largest bound). Four rounds over 8-bit digits, most
// significant first, each a histogram of the keys that still match the
// digits found so far, give the key tau of the need-th smallest key and the
// number `take` of keys equal to tau that belong to the selection. The
// selection is every key below tau and the `take` lowest-indexed keys equal
// to tau: exactly the first min(K, non-empty) blocks under (bound
// descending, index ascending). A prefix count gives each its slot in
// ascending block order.
constexpr uint32_t EMPTY = 0xffffffffu;           // key of an empty block

__global__ void __launch_bounds__(SORT_THREADS) k_topk_pick(TopkArgs a, const __grid_constant__ NfTable nt) {
    extern __shared__ uint32_t key[];              // [nf]
    __shared__ int hist[256];
    __shared__ int ws[32];
    __shared__ int s_digit, s_below;
    // the decode may be scheduled now; it waits for the selection
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u = blockIdx.x, tid = threadIdx.x, nth = blockDim.x, n = unit_nf(a, nt, u);
    const float *bd = a.bound + (size_t)u * a.NB;
    // a contiguous chunk of blocks per thread, so that prefix counts follow block order
    const int chunk = (n + nth - 1) / nth, jb = min(n, tid * chunk), je = min(n, jb + chunk);
    // the bounds are the previous grid's results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    int ne_local = 0;
    for (int j = jb; j < je; ++j) {
        const float f = bd[j];
        const bool nonempty = f != -CUDART_INF_F;
        key[j] = nonempty ? ~ordered(f) : EMPTY;   // a finite bound never maps to EMPTY
        ne_local += nonempty;
    }
    int ne;
    block_exscan(ne_local, ws, ne);
    const int want = min(a.K, ne);
    uint32_t prefix = 0, mask = 0;
    int need = want;
    for (int shift = 24; shift >= 0 && want > 0; shift -= 8) {
        for (int i = tid; i < 256; i += nth) hist[i] = 0;
        __syncthreads();
        for (int j = jb; j < je; ++j) {
            const uint32_t k = key[j];
            if (k != EMPTY && (k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l owns digits 8l .. 8l+7
            int cnt[8], sum = 0;
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                cnt[x] = hist[8 * tid + x];
                sum += cnt[x];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (tid >= o) incl += y;
            }
            const int excl = incl - sum;
            if (excl < need && need <= incl) {   // exactly one lane
                int c = excl, dg = 8 * tid;
#pragma unroll
                for (int x = 0; x < 8; ++x) {
                    if (c + cnt[x] >= need) {
                        dg = 8 * tid + x;
                        break;
                    }
                    c += cnt[x];
                }
                s_digit = dg;
                s_below = c;
            }
        }
        __syncthreads();
        prefix |= (uint32_t)s_digit << shift;
        mask |= 255u << shift;
        need -= s_below;
        __syncthreads();
    }
    // keys equal to tau = prefix: the `need` lowest-indexed ones are taken
    int eq_local = 0;
    for (int j = jb; j < je; ++j) eq_local += want > 0 && key[j] != EMPTY && key[j] == prefix;
    int eq_total;
    int eq_before = block_exscan(eq_local, ws, eq_total);
    int sel_local = 0;
    for (int j = jb; j < je; ++j) {
        const uint32_t k = key[j];
        const bool ok = want > 0 && k != EMPTY;
        const bool take = ok && (k < prefix || (k == prefix && eq_before++ < need));
        key[j] = take ? 1u : 0u;                   // reused as the selection mark
        sel_local += take;
    }
    int nsel;
    int pos = block_exscan(sel_local, ws, nsel);
    int32_t *out = a.sel + (size_t)u * a.Kc;
    for (int j = jb; j < je; ++j)
        if (key[j]) out[pos++] = j;
    for (int i = nsel + tid; i < a.Kc; i += nth) out[i] = -1;
}

}  // namespace

int topk_smem_bytes(int d, int gs, int nf) {
    (void)d;
    (void)gs;
    return (nf > 1 ? nf : 1) * 4;
}

cudaError_t launch_topk_select(const ott_cache *c, const __half *q, int K, int Kc, cudaStream_t s) {
    TopkArgs a;
    NfTable nt;
    int nf_max = c->nf;
    a.ragged = c->ragged;
    if (c->ragged) {
        nf_max = 0;
        for (int b = 0; b < c->B; ++b) {
            nt.nf[b] = c->nfb[b];
            nf_max = c->nfb[b] > nf_max ? c->nfb[b] : nf_max;
        }
    }
    a.bt = c->paged ? c->bt : nullptr;
    a.blk = c->blk;
    a.blk_bytes = c->blk_bytes;
    a.NB = c->NB;
    a.nf = nf_max;
    a.G = c->G;
    a.P = c->P;
    a.jfull = (c->P + c->G - 1) / c->G;
    a.bcnt = c->bcnt;   // null unless block sizes differ from the norm criterion's
    a.q = q;
    a.Hq = c->Hq;
    a.Hkv = c->Hkv;
    a.g = c->gq;
    a.K = K;
    a.Kc = Kc;
    a.bound = c->bound;
    a.sel = c->sel;
    const dim3 grid((unsigned)((nf_max + BND_BLOCKS - 1) / BND_BLOCKS), (unsigned)c->U);
    bool found = false;
#define OTT_BND(D_, G_)                                                       \
    if (c->d == D_ && c->gs == G_) {                                          \
        k_topk_bounds<D_, G_><<<grid, BND_THREADS, 0, s>>>(a, nt);            \
        found = true;                                                         \
    }
    OTT_BND(128, 1) OTT_BND(128, 2) OTT_BND(128, 4) OTT_BND(64, 1) OTT_BND(64, 2) OTT_BND(64, 4)
#undef OTT_BND
    if (!found) return cudaErrorInvalidValue;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // whole warps, up to SORT_THREADS, about two blocks per thread
    int th = ((nf_max + 1) / 2 + 31) / 32 * 32;
    th = th < 32 ? 32 : (th > SORT_THREADS ? SORT_THREADS : th);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c->U);
    cfg.blockDim = dim3((unsigned)th);
    cfg.dynamicSmemBytes = (size_t)topk_smem_bytes(c->d, c->gq, nf_max);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_topk_pick, a, nt);
}

cudaError_t set_topk_attributes(int d, int gs, int smem_max) {
    (void)d;
    (void)gs;
    return cudaFuncSetAttribute(k_topk_pick, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max - 2048);
}

}  // namespace ott
