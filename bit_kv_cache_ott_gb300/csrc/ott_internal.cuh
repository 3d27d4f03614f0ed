// ott_internal.cuh -- device layout of the OTT cache and the launcher
// interface shared by the library's translation units.
//
// Packed cache layout (one unit = one (sequence, kv head)):
//
//   block j of unit u, at blk + (u*NB + j) * block_bytes:
//     [0, 4d)                 K scale/zero, half2 (s, z) per channel
//     then ntile = ceil(G/16) tiles of 16 token slots, 10d bytes each:
//       [0, 4d)    K codes : 32 lanes x d/32 words, lane-major
//       [4d, 8d)   V codes : same
//       [8d, 10d)  V scale/zero half2, index ((gamma*4 + i)*4 + k)
//   A block holds c_j <= G valid tokens in slots 0..c_j-1 (ascending token
//   index); padding slots carry code 0 and scale/zero 0.
//
// Word format. A 32-bit word carries 16 two-bit codes: eight in the low
// half at bits 2p (p = 0..7) and eight in the high half at bits 16+2p.
// Masking position p < 5 leaves the code at bits 2p of each 16-bit half,
// which as an IEEE fp16 number is the subnormal code * 2^(2p-24); positions
// p = 5..7 do the same after a right shift by 10 (class p-5). So one AND
// (plus one shift per word) turns two codes into an exact fp16x2 operand of
// mma.sync, at a power-of-two "class" scale that the other operand or the
// epilogue removes. Which (token, channel) sits at (lane, word, p, half) is
// fixed by the mma.sync m16n8k16 fragment layouts:
//
//   K (A operand of the score MMA, rows = tokens, k = channels):
//     lane = 4r + i, word w = 2*wp + th, slot q = 8*wp + p,
//     o = q / (d/16), kt = q % (d/16):
//       token slot 16*tile + r + 8*th, channel 16*kt + 2i + 8o + half
//   V (A operand of the PV MMA, rows = channels, k = tokens):
//     lane = 4r + i, word w = 2*wp + tp, slot q = 8*wp + p,
//     rowhalf = q / (d/16), mt = q % (d/16):
//       channel 16*mt + r + 8*rowhalf, token slot 16*tile + 2i + 8*tp + half
//   V scale/zero: (gamma, i, k) holds token slot 16*tile + 2i + (k&1) + 8*(k>>1)
//
// Residual ring: rk, rv [U][G+R][d], token t in slot t mod (G+R).
// Outlier pool:  pk, pv [U][P][d], pnorm [U][P], pidx [U][P], kept sorted by
// (norm, token index) ascending; n_pool = min(P, nf*G) for every unit.
// Paged pool (ott_create_paged): block j of unit u lives at pool slot
// bt[u][j] instead of u*NB + j.
// Cold pool (cold-pool policy only): ck, cv [U][C][d], cidx [U][C], a ring
// used first in, first out, with (count, slot of the oldest) in cmeta [U][2];
// block sizes then depend on the data and are kept in bcnt [U][NB].
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/ott.h"

namespace ott {

constexpr int TILE = 16;          // token slots per tile
constexpr int CHUNK_TILES = 4;    // tiles per staged chunk in the decode kernel
constexpr int DEC_WARPS = 16;     // warps per decode CTA
constexpr int FP16_CHUNK = 16;    // fp16 tokens per decode work item
constexpr int RAGGED_MAX = 256;   // sequences in a cache whose sequences may differ in length

__host__ __device__ constexpr int ksz_bytes(int d) { return 4 * d; }
__host__ __device__ constexpr int tile_bytes(int d) { return 10 * d; }
__host__ __device__ constexpr int tile_k_off(int) { return 0; }
__host__ __device__ constexpr int tile_v_off(int d) { return 4 * d; }
__host__ __device__ constexpr int tile_sz_off(int d) { return 8 * d; }
__host__ __device__ constexpr int stage_bytes(int d) { return ksz_bytes(d) + CHUNK_TILES * tile_bytes(d); }
__host__ __device__ inline int ntiles_of(int G) { return (G + TILE - 1) / TILE; }
// quantized decode work items per block: chunks of CHUNK_TILES tiles
__host__ __device__ inline int chunks_per_block(int G) {
    return (G + CHUNK_TILES * TILE - 1) / (CHUNK_TILES * TILE);
}
__host__ __device__ inline long long block_bytes_of(int d, int G) {
    return ksz_bytes(d) + (long long)ntiles_of(G) * tile_bytes(d);
}
__host__ __device__ constexpr int cls_of_pos(int p) { return p < 5 ? p : p - 5; }

// Pool size after nf flushes and valid tokens of block j (same for all units).
// Norm criterion (pct < 0): min(nf * G, P). Channel-conditioned criterion
// (pct = p in units of 1/10000): x_j = min(P, ceil(p * (x_{j-1} + G))); the
// map is nondecreasing and x_1 >= x_0 = 0, so the sizes never shrink and stay
// fixed from the first repeat on (at most P + 1 steps).
__host__ __device__ inline int pool_after(int P, int G, long long nf, int pct = -1) {
    if (pct < 0) {
        long long x = nf * (long long)G;
        return (int)(x < P ? x : P);
    }
    int x = 0;
    for (long long j = 0; j < nf; ++j) {
        const long long m = ((long long)pct * (x + G) + 9999) / 10000;
        const int y = (int)(m < P ? m : P);
        if (y == x) break;
        x = y;
    }
    return x;
}
__host__ __device__ inline int block_count(int P, int G, int j, int pct = -1) {
    return pool_after(P, G, j, pct) + G - pool_after(P, G, j + 1, pct);
}

// (token slot t, channel ch) -> (word index lane*(d/32)+w within the tile's
// K region, bit offset). Inverse of the K mapping above.
__host__ __device__ inline void k_loc(int t, int ch, int d, int &word, int &bit) {
    const int nkt = d / 16, nw = d / 32;
    const int tin = t & 15, r = tin & 7, th = tin >> 3;
    const int kt = ch >> 4, rem = ch & 15, o = rem >> 3, i = (rem & 7) >> 1, half = rem & 1;
    const int q = o * nkt + kt, wp = q >> 3, p = q & 7;
    word = (4 * r + i) * nw + 2 * wp + th;
    bit = 16 * half + 2 * p;
}

__host__ __device__ inline void v_loc(int t, int ch, int d, int &word, int &bit) {
    const int nkt = d / 16, nw = d / 32;
    const int tin = t & 15, tp = tin >> 3, i = (tin & 7) >> 1, half = tin & 1;
    const int mt = ch >> 4, rem = ch & 15, rowhalf = rem >> 3, r = rem & 7;
    const int q = rowhalf * nkt + mt, wp = q >> 3, p = q & 7;
    word = (4 * r + i) * nw + 2 * wp + tp;
    bit = 16 * half + 2 * p;
}

__host__ __device__ inline int vsz_index(int t, int gamma) {
    const int tin = t & 15, i = (tin & 7) >> 1, k = (tin & 1) + 2 * (tin >> 3);
    return (gamma * 4 + i) * 4 + k;
}

}  // namespace ott

struct ott_cache {
    int B, Hq, Hkv, d, G, R, P, max_tokens;
    int U, gq, ring, NB, ntile;
    // The decode kernels serve gs query heads of a kv head per pass (1, 2 or
    // 4); a kv head with gq = Hq / Hkv heads is read in S = ceil(gq / gs)
    // passes ("slices"), the last one padded with copies of its last head.
    int gs, S;
    long long blk_bytes;
    long long T;
    int nf;
    int poisoned;
    // no flush (or anything else that writes blocks) queued since the last
    // decode: the next decode may be launched as a programmatic dependent
    int blocks_settled;
    int device;
    int sm_count;
    int flush_smem;
    int maxu;               // units (kv-head slices) one decode warp's item range can touch
    // device memory (one allocation)
    void *mem;
    size_t mem_bytes;
    uint8_t *blk;           // [U][NB][blk_bytes]
    int32_t *bidx;          // [U][NB][G]
    __half *rk, *rv;        // [U][ring][d]
    __half *pk, *pv;        // [U][P][d]
    float *pnorm;           // [U][P]
    int32_t *pidx;          // [U][P]
    float *part;            // [warps][maxu][2][gs][d+2] split-K partials
    int *ctl;               // [1] status flag set by a bounded wait that timed out
    __half *qdev;           // [B][Hq][d] the queries of a step fed from host memory
    // sequences of different lengths (ott_create_ragged + ott_prefill_lens)
    int ragged_capable;     // partials sized for ragged decode
    int ragged;             // per-sequence lengths in effect
    int maxu_r;             // units a decode warp's range can touch in a ragged batch
    std::vector<long long> Tb;   // [B] tokens of each sequence (ragged)
    std::vector<int> nfb;        // [B] flushes of each sequence (ragged)
    // cold-pool policy (ott_create_cold): displaced pool tokens enter a
    // first-in-first-out fp16 pool of `cold` slots instead of the new block
    int cold;               // capacity C, or -1 (displaced tokens are written back)
    __half *ck, *cv;        // [U][C][d]
    int32_t *cidx;          // [U][C]
    int *cmeta;             // [U][2]: tokens in the cold pool, slot of the oldest
    int32_t *bcnt;          // [U][NB] valid tokens of each block (cold-pool or channel criterion)
    // channel-conditioned outlier criterion (ott_create_pct): p in units of
    // 1/10000 (-1: the norm criterion) and the outlier channels per flush
    int pct, n_oc;
    // paged block pool (ott_create_paged): the quantized blocks of all units
    // come from one pool; a flush takes a free slot, a released sequence
    // returns its slots
    int paged;
    int pool_blocks;
    int32_t *bt;            // [U][NB] pool slot of block j of unit u
    int32_t *fstack;        // [pool_blocks] free slots
    int *ftop;              // [1] number of free slots on the stack
    long long free_blocks;  // host mirror of *ftop
    // Top-K sparse decode (ott_decode_attn_topk)
    int32_t *sel;           // [U][Kc] the blocks selected by the last call
    float *bound;           // [U][NB] scratch: the blocks' score bounds
    int topk_ok;            // the selection kernel's shared memory fits for NB blocks
};

namespace ott {

// One sequence of a ragged batch as the decode kernels see it: its work
// items start at `base` (items of unit b*Hkv + h at base + h*Iu), and its
// counts. e[B].base holds the total item count.
struct SeqEntry {
    long long base;
    int nf, ntail, npool, ring_start, Sf, Iu;
};
struct SeqTable {
    SeqEntry e[RAGGED_MAX + 1];
};
// Sequences to flush in one launch (ragged batches): sequence lb[i], group lj[i].
struct FlushList {
    int n;
    int lb[RAGGED_MAX], lj[RAGGED_MAX];
};

// qsrc (optional): the step's queries, copied to c->qdev by the same kernel
cudaError_t launch_append(const ott_cache *c, const __half *k, const __half *v, cudaStream_t s,
                          const __half *qsrc = nullptr);
cudaError_t launch_append_ragged(const ott_cache *c, const __half *k, const __half *v, cudaStream_t s,
                                 const __half *qsrc = nullptr);
cudaError_t launch_flush(const ott_cache *c, const __half *srcK, const __half *srcV,
                         long long src_unit_stride, long long src_mod, long long t0, int j,
                         cudaStream_t s);
cudaError_t launch_flush_list(const ott_cache *c, const __half *srcK, const __half *srcV,
                              long long src_unit_stride, long long src_mod, const FlushList &fl,
                              cudaStream_t s);
cudaError_t launch_copy_tail(const ott_cache *c, const __half *K, const __half *V, int L,
                             long long t_begin, cudaStream_t s);
cudaError_t launch_copy_tail_units(const ott_cache *c, const __half *K, const __half *V, int u0, int nu,
                                   int Lstride, long long t_begin, long long t_end, cudaStream_t s,
                                   int src_u0 = 0);
cudaError_t launch_flush_list_src(const ott_cache *c, const __half *srcK, const __half *srcV,
                                  long long src_unit_stride, long long src_mod, int src_u0, const FlushList &fl,
                                  cudaStream_t s);
cudaError_t launch_release(const ott_cache *c, int b, cudaStream_t s);
// Parallel prefill of units [u0, u0 + nu), nf flushes each, from a source
// holding unit u at (u - src_u0) * src_unit_stride; scratch of
// prefill_scratch_bytes(c, nu, nf) bytes on the device.
bool prefill_parallel_ok(const ott_cache *c, int nf, int shared_units);
size_t prefill_scratch_bytes(const ott_cache *c, int nu, int nf);
cudaError_t launch_prefill_parallel(const ott_cache *c, const __half *srcK, const __half *srcV,
                                    long long src_unit_stride, int src_u0, int u0, int nu, int nf,
                                    uint64_t *scratch, cudaStream_t s);
cudaError_t launch_decode(const ott_cache *c, const __half *q, __half *out, cudaStream_t s);
cudaError_t launch_decode_topk(const ott_cache *c, const __half *q, __half *out, int Kc, cudaStream_t s);
cudaError_t launch_topk_select(const ott_cache *c, const __half *q, int K, int Kc, cudaStream_t s);
int topk_smem_bytes(int d, int gs, int nf);
cudaError_t set_topk_attributes(int d, int gs, int smem_max);
cudaError_t launch_export(const ott_cache *c, int u0, int nu, int nf, uint8_t *stage, cudaStream_t s);
size_t export_stage_bytes(const ott_cache *c, int nu, int nf);
int flush_smem_bytes(int d, int G, int P);
int decode_smem_bytes(int d, int gs);
cudaError_t set_kernel_attributes(int d, int gs, int smem_max);
cudaError_t set_flush_attributes(int d, int smem);
bool decode_supported(int d);
// query heads per decode pass for gq query heads per kv head
inline int slice_heads(int gq) { return (gq == 1 || gq == 2 || gq == 4) ? gq : 4; }

}  // namespace ott
