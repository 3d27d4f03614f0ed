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
//   k_topk_sort: a CTA per unit, one thread per compare-exchange. The blocks'
//     (bound, index) keys are sorted by a bitonic network in shared memory
//     (bound descending, then index); the first min(K, non-empty blocks) are
//     selected and sorted again by index, and written to sel[u][0..Kc) (-1 in
//     the slots left over).
#include <math_constants.h>

#include "ott_internal.cuh"

namespace ott {
namespace {

constexpr int BND_BLOCKS = 32;      // blocks per bounds CTA
constexpr int BND_THREADS = 128;
constexpr int SORT_THREADS = 512;   // at most

struct TopkArgs {
    const uint8_t *blk;
    long long blk_bytes;
    int NB, nf, G, P, jfull;
    const int32_t *bcnt;     // block sizes under the cold-pool policy, else null
    const __half *q;         // [B][Hq][d]
    int Hq, Hkv;
    int K;                   // blocks to keep
    int Kc;                  // slots per unit in sel: min(K, nf)
    float *bound;            // [U][NB] scratch: block bounds
    int32_t *sel;            // [U][Kc]
};

template <int D, int GQ>
__global__ void __launch_bounds__(BND_THREADS) k_topk_bounds(TopkArgs a) {
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
    const int nb = min(BND_BLOCKS, a.nf - j0);
    const int b = u / a.Hkv, hk = u % a.Hkv;
    const __half *qp = a.q + ((size_t)b * a.Hq + hk * GQ) * D;
    for (int e = tid; e < GQ * D; e += nth) qs[e] = __half2float(qp[e]);
    const uint8_t *base = a.blk + ((size_t)u * a.NB + j0) * a.blk_bytes;
    uint4 buf[PER];
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        const int e = tid + i * BND_THREADS, r = e / V4, v = e % V4;
        if (r < nb) buf[i] = __ldg(reinterpret_cast<const uint4 *>(base + (size_t)r * a.blk_bytes) + v);
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
    __syncthreads();
    const int r = tid % BND_BLOCKS, h = tid / BND_BLOCKS;
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
    if (tid < nb) {
        const int j = j0 + tid;
        const int cnt = a.bcnt ? a.bcnt[(size_t)u * a.NB + j] : (j >= a.jfull ? a.G : block_count(a.P, a.G, j));
        float best = -CUDART_INF_F;
        if (cnt > 0)
#pragma unroll
            for (int x = 0; x < GQ; ++x) best = part[x][tid] > best ? part[x][tid] : best;
        a.bound[(size_t)u * a.NB + j] = best;
    }
}

// fp32 -> uint32 whose unsigned order is the float order
__device__ __forceinline__ uint32_t ordered(float f) {
    const uint32_t x = __float_as_uint(f);
    return (x & 0x80000000u) ? ~x : (x | 0x80000000u);
}

// Ascending bitonic sort of n (a power of two) keys in shared memory.
template <typename T>
__device__ void bitonic_sort(T *k, int n) {
    for (int size = 2; size <= n; size <<= 1)
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < n / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool up = (lo & size) == 0;
                const T x = k[lo], y = k[hi];
                if ((x > y) == up) {
                    k[lo] = y;
                    k[hi] = x;
                }
            }
            __syncthreads();
        }
}

__global__ void __launch_bounds__(SORT_THREADS) k_topk_sort(TopkArgs a, int n2) {
    extern __shared__ unsigned long long keys[];   // [n2]
    int *idx = reinterpret_cast<int *>(keys + n2);  // [n2]: the selected blocks, then in index order
    // the decode may be scheduled now; it waits for the selection
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u = blockIdx.x, tid = threadIdx.x, nth = blockDim.x;
    const float *bd = a.bound + (size_t)u * a.NB;
    // the bounds are the previous grid's results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // key: (bound descending, index ascending) as one ascending 64-bit key;
    // empty blocks (bound -inf) and padding sort last
    for (int j = tid; j < n2; j += nth) {
        unsigned long long key = ~0ull;
        if (j < a.nf) {
            const float f = bd[j];
            if (f != -CUDART_INF_F) key = ((unsigned long long)(~ordered(f)) << 32) | (unsigned)j;
        }
        keys[j] = key;
    }
    __syncthreads();
    bitonic_sort(keys, n2);
    // the selected blocks, then in ascending order (m2: a power of two >= Kc, <= n2)
    int m2 = 1;
    while (m2 < a.Kc) m2 <<= 1;
    for (int i = tid; i < m2; i += nth) {
        const unsigned long long key = i < a.Kc ? keys[i] : ~0ull;
        idx[i] = key == ~0ull ? 0x7fffffff : (int)(unsigned)(key & 0xffffffffull);
    }
    __syncthreads();
    bitonic_sort(idx, m2);
    int32_t *out = a.sel + (size_t)u * a.Kc;
    for (int i = tid; i < a.Kc; i += nth) out[i] = idx[i] == 0x7fffffff ? -1 : idx[i];
}

int pow2_at_least(int n) {
    int p = 1;
    while (p < n) p <<= 1;
    return p;
}

}  // namespace

int topk_smem_bytes(int d, int gq, int nf) {
    (void)d;
    (void)gq;
    const int n2 = pow2_at_least(nf > 1 ? nf : 1);
    return n2 * 8 + n2 * 4;
}

cudaError_t launch_topk_select(const ott_cache *c, const __half *q, int K, int Kc, cudaStream_t s) {
    TopkArgs a;
    a.blk = c->blk;
    a.blk_bytes = c->blk_bytes;
    a.NB = c->NB;
    a.nf = c->nf;
    a.G = c->G;
    a.P = c->P;
    a.jfull = (c->P + c->G - 1) / c->G;
    a.bcnt = c->cold >= 0 ? c->bcnt : nullptr;
    a.q = q;
    a.Hq = c->Hq;
    a.Hkv = c->Hkv;
    a.K = K;
    a.Kc = Kc;
    a.bound = c->bound;
    a.sel = c->sel;
    const dim3 grid((unsigned)((c->nf + BND_BLOCKS - 1) / BND_BLOCKS), (unsigned)c->U);
    bool found = false;
#define OTT_BND(D_, G_)                                                       \
    if (c->d == D_ && c->gq == G_) {                                          \
        k_topk_bounds<D_, G_><<<grid, BND_THREADS, 0, s>>>(a);                \
        found = true;                                                         \
    }
    OTT_BND(128, 1) OTT_BND(128, 2) OTT_BND(128, 4) OTT_BND(64, 1) OTT_BND(64, 2) OTT_BND(64, 4)
#undef OTT_BND
    if (!found) return cudaErrorInvalidValue;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int n2 = pow2_at_least(c->nf > 1 ? c->nf : 1);
    // one thread per compare-exchange (n2 / 2), whole warps, at most SORT_THREADS
    const int th = n2 / 2 < 32 ? 32 : (n2 / 2 > SORT_THREADS ? SORT_THREADS : n2 / 2);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)c->U);
    cfg.blockDim = dim3((unsigned)th);
    cfg.dynamicSmemBytes = (size_t)topk_smem_bytes(c->d, c->gq, c->nf);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_topk_sort, a, n2);
}

cudaError_t set_topk_attributes(int d, int gq, int smem_max) {
    (void)d;
    (void)gq;
    return cudaFuncSetAttribute(k_topk_sort, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
}

}  // namespace ott
