// ott_api.cu -- the C ABI: argument and state checks, device memory, the
// host-side mirror of the counts (T, nf) and the flush schedule.
//
// The host knows T for every call, so whether an append triggers a flush
// ("every G tokens", zijie-tian.site sec. 3.1; the R newest tokens stay fp16,
// sec. 3.3) is decided here, with no device round trip on the decode path.
#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "ott_internal.cuh"

using namespace ott;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int fail_cuda(ott_cache *c, cudaError_t e) {
    if (e == cudaSuccess) return OTT_OK;
    if (c) c->poisoned = 1;
    return OTT_ERR_CUDA;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Flush needed after T tokens with nf flushes done?
bool flush_due(const ott_cache *c) { return c->T - (long long)c->nf * c->G >= (long long)c->G + c->R; }
bool flush_due_seq(const ott_cache *c, int b) {
    return c->Tb[b] - (long long)c->nfb[b] * c->G >= (long long)c->G + c->R;
}
int flushes_after(const ott_cache *c, long long T) { return T >= c->G + c->R ? (int)((T - c->R) / c->G) : 0; }

int create_cache(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens, int ragged,
                 int cold, ott_cache **out, long long pool_blocks = 0, int pct = -1, int n_oc = 0);

// Paged pool: blocks that flushes of these sequences (group j of sequence b
// for j in [nf_from[b], nf_to[b])) need. 0 for a cache without the pool.
long long blocks_needed(const ott_cache *c, long long n_unit_flushes) { return c->paged ? n_unit_flushes : 0; }

// Ragged caches: every sequence must hold a token for appends and decodes
// (except at the very start, T = 0, when all sequences grow together).
bool some_sequence_empty(const ott_cache *c) {
    if (!c->ragged || c->T == 0) return false;
    for (int b = 0; b < c->B; ++b)
        if (c->Tb[b] == 0) return true;
    return false;
}

// With per-sequence counts, T is the longest sequence: releases and refills
// move it both ways, and the capacity checks are per sequence.
void refresh_T(ott_cache *c) {
    long long t = 0;
    for (int b = 0; b < c->B; ++b) t = c->Tb[b] > t ? c->Tb[b] : t;
    c->T = t;
}

// Switch a cache to per-sequence counts (ragged decode and flush lists),
// every sequence at the current uniform count.
void to_per_sequence(ott_cache *c) {
    c->Tb.assign(c->B, c->T);
    c->nfb.assign(c->B, c->nf);
    c->ragged = 1;
    c->nf = 0;
}

// Every flush of units [u0, u0 + nu), nf each, in one parallel pass (the
// source holds unit u at (u - src_u0) * unit_stride). False when the policy
// needs the flushes one after another, when the call runs one pass per
// sequence and its group-by-group launches would carry enough units
// (shared_units; 0 for a call with a single pass) to fill the GPU, or when
// no scratch could be had: the caller then flushes group by group.
// The parallel prefill's scratch comes from a stream-ordered pool that the
// library creates once per device and that keeps up to kScratchKeep bytes
// between calls: with the default pool's threshold of zero, every prefill
// after a synchronization would map its scratch afresh (about 0.1 ms of host
// time before the first kernel). If this pool cannot be had or used (for
// example after a device reset), the device's default pool serves.
constexpr uint64_t kScratchKeep = 1ull << 30;
constexpr int kMaxDevices = 64;

cudaMemPool_t scratch_pool(int dev) {
    static std::mutex mu;
    static cudaMemPool_t pools[kMaxDevices] = {};
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.handleTypes = cudaMemHandleTypeNone;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t p = nullptr;
        if (cudaMemPoolCreate(&p, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = kScratchKeep;
        if (cudaMemPoolSetAttribute(p, cudaMemPoolAttrReleaseThreshold, &keep) != cudaSuccess) cudaGetLastError();
        pools[dev] = p;
    }
    return pools[dev];
}

bool try_prefill_parallel(const ott_cache *c, const __half *K, const __half *V, long long unit_stride, int src_u0,
                          int u0, int nu, int nf, int shared_units, cudaStream_t s, cudaError_t &err) {
    err = cudaSuccess;
    if (!prefill_parallel_ok(c, nf, shared_units)) return false;
    void *scratch = nullptr;
    const size_t bytes = prefill_scratch_bytes(c, nu, nf);
    const cudaMemPool_t pool = scratch_pool(c->device);
    if (!pool || cudaMallocFromPoolAsync(&scratch, bytes, pool, s) != cudaSuccess) {
        cudaGetLastError();
        scratch = nullptr;
        if (cudaMallocAsync(&scratch, bytes, s) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
    }
    err = launch_prefill_parallel(c, K, V, unit_stride, src_u0, u0, nu, nf, static_cast<uint64_t *>(scratch), s);
    const cudaError_t e2 = cudaFreeAsync(scratch, s);
    if (err == cudaSuccess) err = e2;
    return true;
}

}  // namespace

extern "C" {

const char *ott_status_str(int code) {
    switch (code) {
        case OTT_OK: return "ok";
        case OTT_ERR_INVALID: return "invalid argument";
        case OTT_ERR_STATE: return "call not allowed in the current cache state";
        case OTT_ERR_CAPACITY: return "capacity (max_tokens) exceeded";
        case OTT_ERR_OOM: return "device allocation failed";
        case OTT_ERR_CUDA: return "CUDA error (handle poisoned)";
        case OTT_ERR_DEVICE: return "a kernel timed out on a bounded wait";
        default: return "unknown status";
    }
}

int ott_create(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens, ott_cache **out) {
    return create_cache(B, Hq, Hkv, d, G, R, P, max_tokens, 0, -1, out);
}

int ott_create_cold(int B, int Hq, int Hkv, int d, int G, int R, int P, int C, int max_tokens, ott_cache **out) {
    if (C < 0 || C > OTT_COLD_MAX) {
        if (out) *out = nullptr;
        return OTT_ERR_INVALID;
    }
    return create_cache(B, Hq, Hkv, d, G, R, P, max_tokens, 0, C, out);
}

int ott_create_pct(int B, int Hq, int Hkv, int d, int G, int R, int P, int pct, int n_oc, int max_tokens,
                   ott_cache **out) {
    if (pct < 0 || pct > 10000 || n_oc < 1 || n_oc > d) {
        if (out) *out = nullptr;
        return OTT_ERR_INVALID;
    }
    return create_cache(B, Hq, Hkv, d, G, R, P, max_tokens, 0, -1, out, 0, pct, n_oc);
}

int ott_create_paged(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens, long long pool_blocks,
                     ott_cache **out) {
    if (B > RAGGED_MAX || pool_blocks < 1 || pool_blocks > 0x7fffffffLL) {
        if (out) *out = nullptr;
        return OTT_ERR_INVALID;
    }
    return create_cache(B, Hq, Hkv, d, G, R, P, max_tokens, 1, -1, out, pool_blocks);
}

int ott_create_ragged(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens, ott_cache **out) {
    if (B > RAGGED_MAX) {
        if (out) *out = nullptr;
        return OTT_ERR_INVALID;
    }
    return create_cache(B, Hq, Hkv, d, G, R, P, max_tokens, 1, -1, out);
}

}  // extern "C"

namespace {

int create_cache(int B, int Hq, int Hkv, int d, int G, int R, int P, int max_tokens, int ragged,
                 int cold, ott_cache **out, long long pool_blocks, int pct, int n_oc) {
    if (!out) return OTT_ERR_INVALID;
    *out = nullptr;
    if (B < 1 || Hkv < 1 || Hq < 1 || Hq % Hkv != 0 || G < 1 || R < 0 || P < 0 || max_tokens < 0)
        return OTT_ERR_INVALID;
    const int gq = Hq / Hkv;
    if (!decode_supported(d)) return OTT_ERR_INVALID;
    // query heads per decode pass, and passes (slices) per kv head
    const int gs = slice_heads(gq), S = (gq + gs - 1) / gs;
    if ((long long)B * Hkv * S > INT_MAX / 64 || (long long)B * Hq > INT_MAX / 4 || (long long)G + R + P > (1 << 20))
        return OTT_ERR_INVALID;

    int dev = 0, sms = 0, smem_optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return OTT_ERR_CUDA;
    const int fsmem = flush_smem_bytes(d, G, P);
    if (fsmem > smem_optin || decode_smem_bytes(d, gs) > smem_optin) return OTT_ERR_INVALID;

    ott_cache *c = new (std::nothrow) ott_cache();
    if (!c) return OTT_ERR_OOM;
    c->B = B; c->Hq = Hq; c->Hkv = Hkv; c->d = d; c->G = G; c->R = R; c->P = P;
    c->max_tokens = max_tokens;
    c->U = B * Hkv;
    c->gq = gq;
    c->gs = gs;
    c->S = S;
    c->ring = G + R;
    c->NB = max_tokens >= G + R ? (max_tokens - R) / G : 0;
    c->ntile = ntiles_of(G);
    c->blk_bytes = block_bytes_of(d, G);
    c->device = dev;
    c->sm_count = sms;
    c->flush_smem = fsmem;
    // the decode grid's warps split the work items evenly; a warp's range
    // (at most W/NW + 1 items) touches at most U*S/NW + 2 units (kv-head slices)
    const int nwarps = sms * DEC_WARPS;
    c->maxu = (int)((long long)B * Hkv * S / nwarps) + 2;
    // ragged batches: units differ in length, so a range of L items can touch
    // up to L units; L <= ceil(W_max / warps) with at most NB blocks of
    // chunks_per_block(G) items and ceil((G + R + P) / FP16_CHUNK) fp16 items
    // per unit
    c->ragged_capable = ragged;
    c->ragged = 0;
    c->maxu_r = 0;
    if (ragged) {
        const long long iu_max = (G + R + P + FP16_CHUNK - 1) / FP16_CHUNK + (long long)c->NB * chunks_per_block(G);
        const long long w_max = (long long)B * Hkv * S * iu_max;
        c->maxu_r = (int)((w_max + nwarps - 1) / nwarps) + 2;
        c->Tb.assign(B, 0);
        c->nfb.assign(B, 0);
    }
    const int maxu_alloc = c->maxu > c->maxu_r ? c->maxu : c->maxu_r;

    const size_t U = (size_t)c->U;
    c->paged = pool_blocks > 0;
    c->pool_blocks = (int)pool_blocks;
    c->free_blocks = pool_blocks;
    const size_t sz_blk = (c->paged ? (size_t)pool_blocks : U * c->NB) * (size_t)c->blk_bytes;
    const size_t sz_bt = c->paged ? U * c->NB * 4 : 0, sz_fs = c->paged ? (size_t)pool_blocks * 4 : 0;
    const size_t sz_bidx = U * c->NB * (size_t)G * 4;
    const size_t sz_ring = U * c->ring * (size_t)d * 2;
    const size_t sz_pool = U * (size_t)P * d * 2;
    const size_t sz_pn = U * (size_t)P * 4;
    const size_t sz_part = (size_t)nwarps * maxu_alloc * 2 * gs * (d + 2) * 4;
    c->cold = cold;
    c->pct = pct;
    c->n_oc = n_oc;
    const size_t Cs = cold > 0 ? (size_t)cold : 0;
    const size_t sz_cold = U * Cs * d * 2, sz_cidx = U * Cs * 4;
    const size_t sz_cmeta = cold >= 0 ? U * 8 : 0, sz_bcnt = (cold >= 0 || pct >= 0) ? U * c->NB * 4 : 0;
    const size_t sz_sel = U * c->NB * 4;   // also the size of the bound scratch
    size_t off = 0;
    const size_t o_blk = off; off = round_up(off + sz_blk, 256);
    const size_t o_bidx = off; off = round_up(off + sz_bidx, 256);
    const size_t o_rk = off; off = round_up(off + sz_ring, 256);
    const size_t o_rv = off; off = round_up(off + sz_ring, 256);
    const size_t o_pk = off; off = round_up(off + sz_pool, 256);
    const size_t o_pv = off; off = round_up(off + sz_pool, 256);
    const size_t o_pn = off; off = round_up(off + sz_pn, 256);
    const size_t o_pi = off; off = round_up(off + sz_pn, 256);
    const size_t o_part = off; off = round_up(off + sz_part, 256);
    const size_t o_ctl = off; off = round_up(off + 64, 256);
    const size_t o_q = off; off = round_up(off + (size_t)B * Hq * d * 2, 256);
    const size_t o_ck = off; off = round_up(off + sz_cold, 256);
    const size_t o_cv = off; off = round_up(off + sz_cold, 256);
    const size_t o_ci = off; off = round_up(off + sz_cidx, 256);
    const size_t o_cm = off; off = round_up(off + sz_cmeta, 256);
    const size_t o_bc = off; off = round_up(off + sz_bcnt, 256);
    const size_t o_sel = off; off = round_up(off + sz_sel, 256);
    const size_t o_bt = off; off = round_up(off + sz_bt, 256);
    const size_t o_fs = off; off = round_up(off + sz_fs, 256);
    const size_t o_ft = off; off = round_up(off + 16, 256);
    const size_t o_bnd = off; off = round_up(off + sz_sel, 256);
    c->mem_bytes = off;

    // Host-side fault injection for tests: OTT_FAULT=alloc makes the device
    // allocation report failure (exercises the cleanup path without a GPU fault).
    const char *fault = std::getenv("OTT_FAULT");
    if (fault && std::strcmp(fault, "alloc") == 0) {
        delete c;
        return OTT_ERR_OOM;
    }
    void *mem = nullptr;
    e = cudaMalloc(&mem, c->mem_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        delete c;
        return OTT_ERR_OOM;
    }
    c->mem = mem;
    uint8_t *base = static_cast<uint8_t *>(mem);
    c->blk = base + o_blk;
    c->bidx = reinterpret_cast<int32_t *>(base + o_bidx);
    c->rk = reinterpret_cast<__half *>(base + o_rk);
    c->rv = reinterpret_cast<__half *>(base + o_rv);
    c->pk = reinterpret_cast<__half *>(base + o_pk);
    c->pv = reinterpret_cast<__half *>(base + o_pv);
    c->pnorm = reinterpret_cast<float *>(base + o_pn);
    c->pidx = reinterpret_cast<int32_t *>(base + o_pi);
    c->part = reinterpret_cast<float *>(base + o_part);
    c->ctl = reinterpret_cast<int *>(base + o_ctl);
    c->qdev = reinterpret_cast<__half *>(base + o_q);
    c->ck = sz_cold ? reinterpret_cast<__half *>(base + o_ck) : nullptr;
    c->cv = sz_cold ? reinterpret_cast<__half *>(base + o_cv) : nullptr;
    c->cidx = sz_cidx ? reinterpret_cast<int32_t *>(base + o_ci) : nullptr;
    c->cmeta = sz_cmeta ? reinterpret_cast<int *>(base + o_cm) : nullptr;
    c->bcnt = sz_bcnt ? reinterpret_cast<int32_t *>(base + o_bc) : nullptr;
    c->sel = reinterpret_cast<int32_t *>(base + o_sel);
    c->bt = sz_bt ? reinterpret_cast<int32_t *>(base + o_bt) : nullptr;
    c->fstack = sz_fs ? reinterpret_cast<int32_t *>(base + o_fs) : nullptr;
    c->ftop = reinterpret_cast<int *>(base + o_ft);
    c->bound = reinterpret_cast<float *>(base + o_bnd);
    c->topk_ok = topk_smem_bytes(d, gs, c->NB) <= smem_optin - 2048;
    e = cudaMemset(mem, 0, c->mem_bytes);
    if (e == cudaSuccess) e = set_kernel_attributes(d, gs, smem_optin);
    if (e == cudaSuccess) e = set_topk_attributes(d, gs, smem_optin);
    if (e == cudaSuccess && c->paged) {
        // every pool slot free
        std::vector<int32_t> slots((size_t)pool_blocks);
        for (long long i = 0; i < pool_blocks; ++i) slots[(size_t)i] = (int32_t)i;
        const int top = (int)pool_blocks;
        e = cudaMemcpy(c->fstack, slots.data(), slots.size() * 4, cudaMemcpyHostToDevice);
        if (e == cudaSuccess) e = cudaMemcpy(c->ftop, &top, sizeof(int), cudaMemcpyHostToDevice);
    }
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        cudaFree(mem);
        delete c;
        return OTT_ERR_CUDA;
    }
    *out = c;
    return OTT_OK;
}

}  // namespace

extern "C" {

int ott_destroy(ott_cache *c) {
    if (!c) return OTT_OK;
    cudaError_t e = cudaDeviceSynchronize();
    if (c->mem) {
        cudaError_t e2 = cudaFree(c->mem);
        if (e == cudaSuccess) e = e2;
    }
    delete c;
    return e == cudaSuccess ? OTT_OK : OTT_ERR_CUDA;
}

int ott_prefill(ott_cache *c, const void *K, const void *V, int L, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || c->T != 0) return OTT_ERR_STATE;
    if (L < 0) return OTT_ERR_INVALID;
    if (L > c->max_tokens) return OTT_ERR_CAPACITY;
    if (L == 0) return OTT_OK;
    if (!K || !V || !aligned16(K) || !aligned16(V)) return OTT_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half *Kh = static_cast<const __half *>(K), *Vh = static_cast<const __half *>(V);
    const int nf = L >= c->G + c->R ? (L - c->R) / c->G : 0;
    if (blocks_needed(c, (long long)nf * c->U) > c->free_blocks) return OTT_ERR_CAPACITY;
    c->free_blocks -= blocks_needed(c, (long long)nf * c->U);
    c->blocks_settled = 0;
    cudaError_t e = cudaSuccess;
    if (!try_prefill_parallel(c, Kh, Vh, (long long)L * c->d, 0, 0, c->U, nf, 0, s, e)) {
        for (int j = 0; j < nf && e == cudaSuccess; ++j)
            e = launch_flush(c, Kh, Vh, (long long)L * c->d, LLONG_MAX, (long long)j * c->G, j, s);
    }
    if (e != cudaSuccess) return fail_cuda(c, e);
    e = launch_copy_tail(c, Kh, Vh, L, (long long)nf * c->G, s);
    if (e != cudaSuccess) return fail_cuda(c, e);
    c->T = L;
    c->nf = nf;
    // a paged cache reads blocks through the table, and a cache emptied by
    // releases keeps per-sequence counts: both continue per sequence
    if (c->paged || c->ragged) {
        c->ragged = 0;
        to_per_sequence(c);
    }
    return OTT_OK;
}

int ott_prefill_lens(ott_cache *c, const void *K, const void *V, const int *lens, int Lmax, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (!c->ragged_capable || c->poisoned || c->T != 0) return OTT_ERR_STATE;
    if (!lens || Lmax < 1 || !K || !V || !aligned16(K) || !aligned16(V)) return OTT_ERR_INVALID;
    if (Lmax > c->max_tokens) return OTT_ERR_CAPACITY;
    int nf_max = 0;
    long long unit_flushes = 0;
    for (int b = 0; b < c->B; ++b) {
        if (lens[b] < 1 || lens[b] > Lmax) return OTT_ERR_INVALID;
        const int nf = flushes_after(c, lens[b]);
        nf_max = nf > nf_max ? nf : nf_max;
        unit_flushes += (long long)nf * c->Hkv;
    }
    if (blocks_needed(c, unit_flushes) > c->free_blocks) return OTT_ERR_CAPACITY;
    c->free_blocks -= blocks_needed(c, unit_flushes);
    c->blocks_settled = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half *Kh = static_cast<const __half *>(K), *Vh = static_cast<const __half *>(V);
    // each sequence in one parallel pass where it can; the rest group by
    // group, every such sequence's group j in one launch
    std::vector<char> done(c->B, 0);
    for (int b = 0; b < c->B; ++b) {
        cudaError_t e = cudaSuccess;
        done[b] = try_prefill_parallel(c, Kh, Vh, (long long)Lmax * c->d, 0, b * c->Hkv, c->Hkv,
                                       flushes_after(c, lens[b]), c->U, s, e);
        if (e != cudaSuccess) return fail_cuda(c, e);
    }
    for (int j = 0; j < nf_max; ++j) {
        FlushList fl;
        fl.n = 0;
        for (int b = 0; b < c->B; ++b)
            if (!done[b] && flushes_after(c, lens[b]) > j) {
                fl.lb[fl.n] = b;
                fl.lj[fl.n] = j;
                ++fl.n;
            }
        if (fl.n == 0) break;
        cudaError_t e = launch_flush_list(c, Kh, Vh, (long long)Lmax * c->d, LLONG_MAX, fl, s);
        if (e != cudaSuccess) return fail_cuda(c, e);
    }
    long long Tmax = 0;
    for (int b = 0; b < c->B; ++b) {
        const int nf = flushes_after(c, lens[b]);
        cudaError_t e = launch_copy_tail_units(c, Kh, Vh, b * c->Hkv, c->Hkv, Lmax, (long long)nf * c->G,
                                               lens[b], s);
        if (e != cudaSuccess) return fail_cuda(c, e);
        c->Tb[b] = lens[b];
        c->nfb[b] = nf;
        Tmax = lens[b] > Tmax ? lens[b] : Tmax;
    }
    c->ragged = 1;
    c->T = Tmax;
    c->nf = 0;
    return OTT_OK;
}

namespace {

int append_ragged(ott_cache *c, const __half *k, const __half *v, cudaStream_t s, const __half *qsrc) {
    long long due = 0;   // sequences whose residual window fills with this token
    for (int b = 0; b < c->B; ++b)
        due += c->Tb[b] + 1 - (long long)c->nfb[b] * c->G >= (long long)c->G + c->R;
    if (blocks_needed(c, due * c->Hkv) > c->free_blocks) return OTT_ERR_CAPACITY;
    c->free_blocks -= blocks_needed(c, due * c->Hkv);
    cudaError_t e = launch_append_ragged(c, k, v, s, qsrc);
    if (e != cudaSuccess) return fail_cuda(c, e);
    FlushList fl;
    fl.n = 0;
    for (int b = 0; b < c->B; ++b) {
        c->Tb[b] += 1;
        if (flush_due_seq(c, b)) {
            fl.lb[fl.n] = b;
            fl.lj[fl.n] = c->nfb[b];
            ++fl.n;
        }
    }
    c->T += 1;
    if (fl.n > 0) c->blocks_settled = 0;
    e = launch_flush_list(c, c->rk, c->rv, (long long)c->ring * c->d, c->ring, fl, s);
    if (e != cudaSuccess) return fail_cuda(c, e);
    for (int i = 0; i < fl.n; ++i) c->nfb[fl.lb[i]] += 1;
    return OTT_OK;
}

}  // namespace

namespace {

// The append of ott_append and ott_step_host (qsrc: the step's queries to
// copy to c->qdev in the same kernel, or null). Arguments are checked.
int append_impl(ott_cache *c, const void *k, const void *v, cudaStream_t s, const __half *qsrc) {
    // with per-sequence counts T is the longest sequence, so this is each
    // sequence's own capacity check
    if (c->T + 1 > c->max_tokens) return OTT_ERR_CAPACITY;
    if (some_sequence_empty(c)) return OTT_ERR_STATE;
    if (c->paged && !c->ragged) to_per_sequence(c);   // blocks are read through the table
    if (c->ragged)
        return append_ragged(c, static_cast<const __half *>(k), static_cast<const __half *>(v), s, qsrc);
    const bool due = c->T + 1 - (long long)c->nf * c->G >= (long long)c->G + c->R;
    if (due && blocks_needed(c, c->U) > c->free_blocks) return OTT_ERR_CAPACITY;
    if (due) c->free_blocks -= blocks_needed(c, c->U);
    cudaError_t e = launch_append(c, static_cast<const __half *>(k), static_cast<const __half *>(v), s, qsrc);
    if (e != cudaSuccess) return fail_cuda(c, e);
    c->T += 1;
    if (flush_due(c)) {
        c->blocks_settled = 0;
        e = launch_flush(c, c->rk, c->rv, (long long)c->ring * c->d, c->ring, (long long)c->nf * c->G, c->nf, s);
        if (e != cudaSuccess) return fail_cuda(c, e);
        c->nf += 1;
    }
    return OTT_OK;
}

// The device address of pinned host memory (null if it is not mapped pinned memory).
const void *mapped(const void *host) {
    void *d = nullptr;
    if (!host || cudaHostGetDevicePointer(&d, const_cast<void *>(host), 0) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return d;
}

}  // namespace

int ott_append(ott_cache *c, const void *k, const void *v, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned) return OTT_ERR_STATE;
    if (!k || !v || !aligned16(k) || !aligned16(v)) return OTT_ERR_INVALID;
    return append_impl(c, k, v, static_cast<cudaStream_t>(stream), nullptr);
}

int ott_step_host(ott_cache *c, const void *k, const void *v, const void *q, void *out, int topk, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned) return OTT_ERR_STATE;
    const void *dk = mapped(k), *dv = mapped(v), *dq = mapped(q);
    void *dout = const_cast<void *>(mapped(out));
    if (!dk || !dv || !dq || !dout || !aligned16(dk) || !aligned16(dv) || !aligned16(dq) || !aligned16(dout))
        return OTT_ERR_INVALID;
    if (out == q || out == k || out == v) return OTT_ERR_INVALID;
    if (topk > 0 && !c->topk_ok) return OTT_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int rc = append_impl(c, dk, dv, s, static_cast<const __half *>(dq));
    if (rc != OTT_OK) return rc;
    if (topk > 0) return ott_decode_attn_topk(c, c->qdev, dout, topk, nullptr, stream);
    const cudaError_t e = launch_decode(c, c->qdev, static_cast<__half *>(dout), s);
    if (e != cudaSuccess) return fail_cuda(c, e);
    c->blocks_settled = 1;
    return OTT_OK;
}

int ott_decode_attn(ott_cache *c, const void *q, void *out, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || c->T < 1 || some_sequence_empty(c)) return OTT_ERR_STATE;
    if (!q || !out || !aligned16(q) || !aligned16(out) || q == out) return OTT_ERR_INVALID;
    cudaError_t e = launch_decode(c, static_cast<const __half *>(q), static_cast<__half *>(out),
                                  static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) c->blocks_settled = 1;
    return fail_cuda(c, e);
}

int ott_decode_attn_topk(ott_cache *c, const void *q, void *out, int K, int32_t *sel, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || c->T < 1 || some_sequence_empty(c)) return OTT_ERR_STATE;
    if (K < 1 || !c->topk_ok || !q || !out || !aligned16(q) || !aligned16(out) || q == out) return OTT_ERR_INVALID;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half *qh = static_cast<const __half *>(q);
    int nf_max = c->nf;
    if (c->ragged)
        for (int b = 0; b < c->B; ++b) nf_max = c->nfb[b] > nf_max ? c->nfb[b] : nf_max;
    const int Kc = K < nf_max ? K : nf_max;
    cudaError_t e = cudaSuccess;
    if (Kc > 0) e = launch_topk_select(c, qh, K, Kc, s);
    if (e == cudaSuccess) e = launch_decode_topk(c, qh, static_cast<__half *>(out), Kc, s);
    if (e == cudaSuccess) c->blocks_settled = 1;
    if (e == cudaSuccess && sel && Kc > 0)
        e = cudaMemcpyAsync(sel, c->sel, (size_t)c->U * Kc * 4, cudaMemcpyDeviceToDevice, s);
    return fail_cuda(c, e);
}

int ott_release_seq(ott_cache *c, int b, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || !c->ragged_capable || c->T < 1) return OTT_ERR_STATE;
    if (b < 0 || b >= c->B) return OTT_ERR_INVALID;
    if (!c->ragged) to_per_sequence(c);   // a uniform prefill so far
    if (c->Tb[b] == 0) return OTT_OK;      // already empty
    c->blocks_settled = 0;
    cudaError_t e = launch_release(c, b, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(c, e);
    c->free_blocks += blocks_needed(c, (long long)c->nfb[b] * c->Hkv);
    c->Tb[b] = 0;
    c->nfb[b] = 0;
    refresh_T(c);
    return OTT_OK;
}

int ott_prefill_seq(ott_cache *c, int b, const void *K, const void *V, int L, void *stream) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || !c->ragged_capable) return OTT_ERR_STATE;
    if (b < 0 || b >= c->B || L < 1 || !K || !V || !aligned16(K) || !aligned16(V)) return OTT_ERR_INVALID;
    if (!c->ragged) {
        if (c->T != 0) return OTT_ERR_STATE;   // a uniform batch: release the sequence first
        to_per_sequence(c);                    // an empty cache filled one sequence at a time
    }
    if (c->Tb[b] != 0) return OTT_ERR_STATE;   // release the sequence first
    if (L > c->max_tokens) return OTT_ERR_CAPACITY;
    const int nf = flushes_after(c, L);
    if (blocks_needed(c, (long long)nf * c->Hkv) > c->free_blocks) return OTT_ERR_CAPACITY;
    c->free_blocks -= blocks_needed(c, (long long)nf * c->Hkv);
    c->blocks_settled = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const __half *Kh = static_cast<const __half *>(K), *Vh = static_cast<const __half *>(V);
    cudaError_t e = cudaSuccess;
    if (!try_prefill_parallel(c, Kh, Vh, (long long)L * c->d, b * c->Hkv, b * c->Hkv, c->Hkv, nf, 0, s, e)) {
        for (int j = 0; j < nf && e == cudaSuccess; ++j) {
            FlushList fl;
            fl.n = 1;
            fl.lb[0] = b;
            fl.lj[0] = j;
            e = launch_flush_list_src(c, Kh, Vh, (long long)L * c->d, LLONG_MAX, b * c->Hkv, fl, s);
        }
    }
    if (e != cudaSuccess) return fail_cuda(c, e);
    e = launch_copy_tail_units(c, Kh, Vh, b * c->Hkv, c->Hkv, L, (long long)nf * c->G, L, s,
                                           b * c->Hkv);
    if (e != cudaSuccess) return fail_cuda(c, e);
    c->Tb[b] = L;
    c->nfb[b] = nf;
    refresh_T(c);
    return OTT_OK;
}

long long ott_free_blocks(const ott_cache *c) {
    if (!c) return OTT_ERR_INVALID;
    return c->paged ? c->free_blocks : -1;
}

int ott_get_seq_counts(const ott_cache *c, int b, long long *T, int *nf, int *tail, int *n_pool) {
    if (!c || b < 0 || b >= c->B) return OTT_ERR_INVALID;
    const long long Tb = c->ragged ? c->Tb[b] : c->T;
    const int nfb = c->ragged ? c->nfb[b] : c->nf;
    if (T) *T = Tb;
    if (nf) *nf = nfb;
    if (tail) *tail = (int)(Tb - (long long)nfb * c->G);
    if (n_pool) *n_pool = pool_after(c->P, c->G, nfb, c->pct);
    return OTT_OK;
}

int ott_get_counts(const ott_cache *c, long long *T, int *nf, int *tail, int *n_pool) {
    if (!c) return OTT_ERR_INVALID;
    if (c->ragged) return ott_get_seq_counts(c, 0, T, nf, tail, n_pool);
    if (T) *T = c->T;
    if (nf) *nf = c->nf;
    if (tail) *tail = (int)(c->T - (long long)c->nf * c->G);
    if (n_pool) *n_pool = pool_after(c->P, c->G, c->nf, c->pct);
    return OTT_OK;
}

int ott_block_count(const ott_cache *c, int j) {
    if (!c) return OTT_ERR_INVALID;
    int nf = c->nf;
    if (c->ragged)
        for (int b = 0; b < c->B; ++b) nf = c->nfb[b] > nf ? c->nfb[b] : nf;
    if (j < 0 || j >= nf) return OTT_ERR_INVALID;
    if (c->cold >= 0) return OTT_ERR_STATE;   // sizes differ per unit: ott_export_cold
    return block_count(c->P, c->G, j, c->pct);
}

long long ott_device_bytes(const ott_cache *c) { return c ? (long long)c->mem_bytes : 0; }

int ott_check_device(ott_cache *c) {
    if (!c) return OTT_ERR_INVALID;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(c, e);
    int flag = 0;
    e = cudaMemcpy(&flag, c->ctl + 1, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(c, e);
    if (!flag) return OTT_OK;
    // a kernel gave up part of its work: the state can no longer be trusted
    c->poisoned = 1;
    return OTT_ERR_DEVICE;
}

int ott_export_state(ott_cache *c, int u0, int nu, const ott_state_export *dst) {
    if (!c || !dst) return OTT_ERR_INVALID;
    if (c->poisoned) return OTT_ERR_STATE;
    if (u0 < 0 || nu < 0 || u0 + nu > c->U) return OTT_ERR_INVALID;
    if (nu == 0) return OTT_OK;
    // a ragged batch is exported one sequence at a time (its units share T and nf)
    if (c->ragged && u0 / c->Hkv != (u0 + nu - 1) / c->Hkv) return OTT_ERR_INVALID;
    const int sb0 = u0 / c->Hkv;
    const long long Tx = c->ragged ? c->Tb[sb0] : c->T;
    const int d = c->d, G = c->G, P = c->P, nf = c->ragged ? c->nfb[sb0] : c->nf;
    const int nt = (int)(Tx - (long long)nf * G);
    const int np = pool_after(P, G, nf, c->pct);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(c, e);

    // blocks: canonical codes and scales through a staging buffer
    if (nf > 0 && (dst->kcode || dst->vcode || dst->ks || dst->kz || dst->vs || dst->vz)) {
        const size_t sb = export_stage_bytes(c, nu, nf);
        uint8_t *stage = nullptr;
        e = cudaMalloc(&stage, sb);
        if (e != cudaSuccess) { cudaGetLastError(); return OTT_ERR_OOM; }
        e = launch_export(c, u0, nu, nf, stage, 0);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        const size_t nblk = (size_t)nu * nf;
        const size_t n_code = nblk * G * (d / 4), n_ksz = nblk * d, n_vsz = nblk * G * (d / 32);
        uint8_t *p = stage;
        if (e == cudaSuccess && dst->kcode) e = cudaMemcpy(dst->kcode, p, n_code, cudaMemcpyDeviceToHost);
        p += n_code;
        if (e == cudaSuccess && dst->vcode) e = cudaMemcpy(dst->vcode, p, n_code, cudaMemcpyDeviceToHost);
        p += n_code;
        if (e == cudaSuccess && dst->ks) e = cudaMemcpy(dst->ks, p, n_ksz * 2, cudaMemcpyDeviceToHost);
        p += n_ksz * 2;
        if (e == cudaSuccess && dst->kz) e = cudaMemcpy(dst->kz, p, n_ksz * 2, cudaMemcpyDeviceToHost);
        p += n_ksz * 2;
        if (e == cudaSuccess && dst->vs) e = cudaMemcpy(dst->vs, p, n_vsz * 2, cudaMemcpyDeviceToHost);
        p += n_vsz * 2;
        if (e == cudaSuccess && dst->vz) e = cudaMemcpy(dst->vz, p, n_vsz * 2, cudaMemcpyDeviceToHost);
        cudaError_t e2 = cudaFree(stage);
        if (e == cudaSuccess) e = e2;
        if (e != cudaSuccess) return fail_cuda(c, e);
    }
    if (nf > 0 && dst->bidx) {
        for (int uu = 0; uu < nu; ++uu) {
            e = cudaMemcpy(dst->bidx + (size_t)uu * nf * G, c->bidx + (size_t)(u0 + uu) * c->NB * G,
                           (size_t)nf * G * 4, cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return fail_cuda(c, e);
        }
    }
    // residual tokens nf*G .. T-1, oldest first
    if (nt > 0 && (dst->tk || dst->tv)) {
        std::vector<uint16_t> rk((size_t)nu * c->ring * d), rv(rk.size());
        e = cudaMemcpy(rk.data(), c->rk + (size_t)u0 * c->ring * d, rk.size() * 2, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess)
            e = cudaMemcpy(rv.data(), c->rv + (size_t)u0 * c->ring * d, rv.size() * 2, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return fail_cuda(c, e);
        for (int uu = 0; uu < nu; ++uu)
            for (int x = 0; x < nt; ++x) {
                const long long t = (long long)nf * G + x;
                const size_t src = ((size_t)uu * c->ring + (size_t)(t % c->ring)) * d;
                const size_t o = ((size_t)uu * nt + x) * d;
                if (dst->tk) std::memcpy(dst->tk + o, rk.data() + src, (size_t)d * 2);
                if (dst->tv) std::memcpy(dst->tv + o, rv.data() + src, (size_t)d * 2);
            }
    }
    // pool in ascending token order
    if (P > 0 && (dst->pidx || dst->pnorm || dst->pk || dst->pv)) {
        const size_t n = (size_t)nu * P;
        std::vector<int32_t> pi(n);
        std::vector<float> pn(n);
        std::vector<uint16_t> pk(n * d), pv(n * d);
        e = cudaMemcpy(pi.data(), c->pidx + (size_t)u0 * P, n * 4, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(pn.data(), c->pnorm + (size_t)u0 * P, n * 4, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(pk.data(), c->pk + (size_t)u0 * P * d, n * d * 2, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(pv.data(), c->pv + (size_t)u0 * P * d, n * d * 2, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return fail_cuda(c, e);
        std::vector<int> ord(P);
        for (int uu = 0; uu < nu; ++uu) {
            for (int x = 0; x < np; ++x) ord[x] = x;
            const int32_t *ip = pi.data() + (size_t)uu * P;
            std::sort(ord.begin(), ord.begin() + np, [&](int a, int b) { return ip[a] < ip[b]; });
            for (int x = 0; x < P; ++x) {
                const bool valid = x < np;
                const size_t so = (size_t)uu * P + (valid ? ord[x] : 0), o = (size_t)uu * P + x;
                if (dst->pidx) dst->pidx[o] = valid ? pi[so] : -1;
                if (dst->pnorm) {
                    uint32_t bits = 0;
                    if (valid) std::memcpy(&bits, &pn[so], 4);
                    dst->pnorm[o] = bits;
                }
                if (dst->pk) {
                    if (valid) std::memcpy(dst->pk + o * d, pk.data() + so * d, (size_t)d * 2);
                    else std::memset(dst->pk + o * d, 0, (size_t)d * 2);
                }
                if (dst->pv) {
                    if (valid) std::memcpy(dst->pv + o * d, pv.data() + so * d, (size_t)d * 2);
                    else std::memset(dst->pv + o * d, 0, (size_t)d * 2);
                }
            }
        }
    }
    return OTT_OK;
}

int ott_export_cold(ott_cache *c, int u0, int nu, int32_t *bcount, int32_t *ncold, int32_t *cidx,
                    uint16_t *ck, uint16_t *cv) {
    if (!c) return OTT_ERR_INVALID;
    if (c->poisoned || c->cold < 0) return OTT_ERR_STATE;
    if (u0 < 0 || nu < 0 || u0 + nu > c->U) return OTT_ERR_INVALID;
    if (nu == 0) return OTT_OK;
    const int d = c->d, C = c->cold, nf = c->nf;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail_cuda(c, e);
    if (bcount && nf > 0)
        for (int uu = 0; uu < nu; ++uu) {
            e = cudaMemcpy(bcount + (size_t)uu * nf, c->bcnt + (size_t)(u0 + uu) * c->NB, (size_t)nf * 4,
                           cudaMemcpyDeviceToHost);
            if (e != cudaSuccess) return fail_cuda(c, e);
        }
    std::vector<int> meta((size_t)nu * 2);
    e = cudaMemcpy(meta.data(), c->cmeta + (size_t)u0 * 2, meta.size() * 4, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda(c, e);
    std::vector<int32_t> ci((size_t)nu * C);
    std::vector<uint16_t> hk((size_t)nu * C * d), hv(hk.size());
    if (C > 0) {
        e = cudaMemcpy(ci.data(), c->cidx + (size_t)u0 * C, ci.size() * 4, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(hk.data(), c->ck + (size_t)u0 * C * d, hk.size() * 2, cudaMemcpyDeviceToHost);
        if (e == cudaSuccess) e = cudaMemcpy(hv.data(), c->cv + (size_t)u0 * C * d, hv.size() * 2, cudaMemcpyDeviceToHost);
        if (e != cudaSuccess) return fail_cuda(c, e);
    }
    for (int uu = 0; uu < nu; ++uu) {
        const int n = C > 0 ? meta[2 * uu] : 0, head = C > 0 ? meta[2 * uu + 1] : 0;
        if (ncold) ncold[uu] = n;
        for (int x = 0; x < C; ++x) {
            const bool valid = x < n;
            const size_t so = (size_t)uu * C + (valid ? (head + x) % C : 0), o = (size_t)uu * C + x;
            if (cidx) cidx[o] = valid ? ci[so] : -1;
            if (ck) {
                if (valid) std::memcpy(ck + o * d, hk.data() + so * d, (size_t)d * 2);
                else std::memset(ck + o * d, 0, (size_t)d * 2);
            }
            if (cv) {
                if (valid) std::memcpy(cv + o * d, hv.data() + so * d, (size_t)d * 2);
                else std::memset(cv + o * d, 0, (size_t)d * 2);
            }
        }
    }
    return OTT_OK;
}

}  // extern "C"
