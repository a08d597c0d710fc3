// Dispatch: per-expert histogram, exclusive scan, stable scatter with capacity mask, payload permute,
// EP-rank-major send layout and the expert FFN's tile schedule.
//
// "v6 长序列和 MoE", table row "dispatch" (group by expert, at most C per expert, pad the rest) and the
// "Capacity" bullet (C = cf*k*T/E, over-capacity tokens dropped; dropless by default in Megatron); the
// follow-up there (sort tokens by expert, run one grouped GEMM). "专家并行" (formulaic), section "All2All":
// the (E, C, M) buffer is pre-sorted by destination expert so that the all-to-all is a block transpose.
//
// Stability and determinism come from a two-level count: the assignments (t, j) in token order are cut
// into chunks of at most 1024; kernel 1 counts each chunk's assignments per expert, kernel 2 (one block)
// scans those counts per expert over the chunks, then over the experts, and writes offsets, kept counts,
// the rank layout and the tile schedule; kernel 3 ranks each assignment inside its chunk (warp match_any
// + per-warp prefix over the chunk's 32 warps) and writes the indices; kernel 4 copies each token row to
// its (at most k) destination rows with 16-byte loads and stores, reading x once. In capacity mode a
// fifth kernel zero-fills the pad rows and marks them -1. For small count tables one launch after the
// count does the scan, the ranking, the copy and the pad fill (dispatch_fused_kernel); its bf16 / fp32 row
// copy goes through the bulk-copy unit (ring_start / ring_finish).
#include <algorithm>
#include <mutex>
#include <cuda_fp8.h>
#include "common.cuh"

namespace moe {

constexpr int kChunkA = 1024;          // assignments per chunk (one thread each)

// Bulk-copy (TMA) unit, untiled: a row piece global -> shared completing on an mbarrier, shared -> global in
// bulk groups of the issuing thread. Addresses and sizes are multiples of 16 bytes.
__device__ __forceinline__ uint32_t shared_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void ring_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void ring_store(void* dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 ::"l"(reinterpret_cast<uint64_t>(dst)), "r"(src), "r"(bytes) : "memory");
}
// Bounded wait for a stage's load: at most `limit` non-blocking polls 32 ns apart; false when they ran out.
constexpr long long kRingDrainLimit = 1LL << 24;
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity, long long limit) {
    for (long long i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
        __nanosleep(32);
    }
    return false;
}

// One thread copies ntok consecutive rows of row_bytes (a multiple of 16) from src to the destination rows
// dest[tl * k + j] >= 0 of dst, piece by piece (pieces of at most SB bytes) through a ring of NS >= 2 shared
// stages. ring_start initialises the stages' mbarriers and puts the first min(NS, pieces) loads in flight;
// ring_finish then stores every piece to its k destinations as one bulk
// group as soon as it has landed, refilling a stage once the group stored out of it has been read. A load that
// does not arrive within `limit` polls latches a timeout; the loads still in flight are then waited for (up to
// kRingDrainLimit polls each, whatever `limit` is, so that none lands in shared memory after the block has
// exited) and the copy stops. If one of those drain waits runs out as well, site 0x111 is latched: that load may
// still land in the shared memory of a block that has exited.
struct RingCursor {
    const char* src;
    uint32_t row_bytes, SB, ring, bars;
    int NS, n;                 // stages, pieces
    int lt, lst, loaded;       // next piece to load: token, stage; pieces loaded so far
    uint32_t loff;             // its byte offset in the row
};

__device__ __forceinline__ void ring_load_next(RingCursor& c) {
    ring_load(c.ring + (uint32_t)c.lst * c.SB, c.src + (size_t)c.lt * c.row_bytes + c.loff,
              min(c.SB, c.row_bytes - c.loff), c.bars + 8u * c.lst);
    c.loff += c.SB;
    if (c.loff >= c.row_bytes) { c.loff = 0; ++c.lt; }
    if (++c.lst == c.NS) c.lst = 0;
    ++c.loaded;
}

__device__ RingCursor ring_start(const char* __restrict__ src, uint32_t row_bytes, int ntok, uint32_t ring,
                                 uint32_t bars, int NS, uint32_t SB) {
    RingCursor c{src, row_bytes, SB, ring, bars, NS, ntok * (int)((row_bytes + SB - 1) / SB), 0, 0, 0, 0u};
    for (int st = 0; st < NS; ++st)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bars + 8u * st) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    while (c.loaded < min(NS, c.n)) ring_load_next(c);
    return c;
}

__device__ void ring_finish(RingCursor& c, int k, const int* __restrict__ dest, char* __restrict__ dst,
                            long long limit, unsigned* err) {
    // store cursor: piece i (token ct, offset coff) sits in stage cst, its load completing phase parity par
    int ct = 0, cst = 0;
    uint32_t coff = 0, par = 0;
    for (int i = 0; i < c.n; ++i) {
        if (!ring_wait(c.bars + 8u * cst, par, limit)) {
            latch_device_error(err, kDevErrTimeout, 0x110u);
            for (int q = i; q < c.loaded; ++q)
                if (!ring_wait(c.bars + 8u * (q % c.NS), (uint32_t)(q / c.NS) & 1u, kRingDrainLimit))
                    latch_device_error(err, kDevErrTimeout, 0x111u);   // a load may still land after the exit
            break;
        }
        const uint32_t bytes = min(c.SB, c.row_bytes - coff);
        const uint32_t from = c.ring + (uint32_t)cst * c.SB;
        for (int j = 0; j < k; ++j) {
            const int d = dest[ct * k + j];
            if (d >= 0) ring_store(dst + (size_t)d * c.row_bytes + coff, from, bytes);
        }
        asm volatile("cp.async.bulk.commit_group;" ::: "memory");
        if (i >= 1 && c.loaded < c.n) {       // refill the stage of piece i - 1 (loaded == i - 1 + NS)
            asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
            ring_load_next(c);
        }
        coff += c.SB;
        if (coff >= c.row_bytes) { coff = 0; ++ct; }
        if (++cst == c.NS) { cst = 0; par ^= 1u; }
    }
    // the stores' sources must have been read before the block's shared memory goes away; their writes complete
    // on their own, and the kernel's end orders them before any later kernel
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Chunk c covers tokens [c * tpc, (c + 1) * tpc), i.e. assignments [c * tpc * k, ...): tpc * k <= kChunkA.
__global__ void __launch_bounds__(kChunkA)
dispatch_count_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int tpc, int32_t* __restrict__ chunk_counts,
                      unsigned* err) {
    extern __shared__ int s_hist[];
    pdl_trigger();                            // the fused dispatch may launch now (it waits for these counts)
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_hist[e] = 0;
    __syncthreads();
    const int a = threadIdx.x;
    const int t = blockIdx.x * tpc + a / k;
    if (a < tpc * k && t < T) {
        const int e = ids[(size_t)blockIdx.x * tpc * k + a];
        if (e >= 0 && e < E) atomicAdd(&s_hist[e], 1);
        else latch_device_error(err, kDevErrBadIndex, 0x100u);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_counts[(size_t)blockIdx.x * E + e] = s_hist[e];
}

// Per-expert kept counts -> offsets, tile prefix (block scans; every thread of the 1024-thread block calls
// it). Thread e < E passes its expert's assignment count n; s_off / s_tp / s_kept receive E + 1 / E + 1 / E
// entries.
__device__ void layout_from_counts(int n, int E, int C, int* s_tmp, int* s_kept, int* s_off, int* s_tp) {
    const int e = threadIdx.x;
    const int kept = (e < E) ? (C > 0 ? min(n, C) : n) : 0;
    const int incl = block_inclusive_scan(kept, s_tmp);
    const int ntiles = (kept + MOE_TILE_M - 1) / MOE_TILE_M;
    const int tincl = block_inclusive_scan(ntiles, s_tmp);
    if (e < E) {
        s_kept[e] = kept;
        s_off[e] = C > 0 ? e * C : incl - kept;
        s_tp[e] = tincl - ntiles;
    }
    if (e == E - 1) { s_off[E] = C > 0 ? E * C : incl; s_tp[E] = tincl; }
    __syncthreads();
}

// Writes offsets, kept counts, the EP rank layout and the tile schedule from the shared layout.
__device__ void publish_layout(int E, int R, const int* s_kept, const int* s_off, const int* s_tp,
                               int32_t* __restrict__ offsets, int32_t* __restrict__ kept_counts,
                               int32_t* __restrict__ rank_counts, int32_t* __restrict__ rank_offsets,
                               int32_t* __restrict__ sched) {
    const int e = threadIdx.x;
    for (int i = e; i <= E; i += blockDim.x) {
        offsets[i] = s_off[i];
        sched[kSchedHeader + i] = s_tp[i];
    }
    if (e < E) kept_counts[e] = s_kept[e];
    if (e == 0) { sched[0] = s_tp[E]; sched[1] = E; }
    const int epr = E / R;
    for (int r = e; r <= R; r += blockDim.x) rank_offsets[r] = s_off[r * epr];
    if (e < R) {
        int sum = 0;
        for (int i = e * epr; i < (e + 1) * epr; ++i) sum += s_kept[i];
        rank_counts[e] = sum;
    }
    if (e < E) {
        int4* tiles = reinterpret_cast<int4*>(sched + sched_tiles_offset(E));
        const int row0 = s_off[e], ntiles = s_tp[e + 1] - s_tp[e];
        for (int m = 0; m < ntiles; ++m) {
            const int rb = row0 + m * MOE_TILE_M;
            tiles[s_tp[e] + m] = make_int4(e, rb, min(rb + MOE_TILE_M, row0 + s_kept[e]), 0);
        }
    }
}

__global__ void __launch_bounds__(1024)
dispatch_scan_kernel(int32_t* __restrict__ chunk_counts /* in: counts, out: per-chunk base */, int nchunks, int E,
                     int C, int R, int32_t* __restrict__ offsets, int32_t* __restrict__ kept_counts,
                     int32_t* __restrict__ rank_counts, int32_t* __restrict__ rank_offsets, int32_t* __restrict__ sched) {
    __shared__ int s_tmp[32];
    __shared__ int s_kept[1024];
    __shared__ int s_off[1025];
    __shared__ int s_tp[1025];
    const int e = threadIdx.x;
    int n = 0;
    if (e < E) {
        for (int c = 0; c < nchunks; ++c) {
            int v = chunk_counts[(size_t)c * E + e];
            chunk_counts[(size_t)c * E + e] = n;
            n += v;
        }
    }
    layout_from_counts(n, E, C, s_tmp, s_kept, s_off, s_tp);
    publish_layout(E, R, s_kept, s_off, s_tp, offsets, kept_counts, rank_counts, rank_offsets, sched);
}

// Ranks the chunk's assignments in token order and writes dest_row, drop_mask, src_token, src_slot.
// s_wc: [32][E] shared scratch; chunk_base(e) = assignments to e in earlier chunks; off = expert offsets.
// Returns the destination row of this thread's assignment (-1: dropped or no assignment).
template <typename Base, typename Off>
__device__ __forceinline__ int rank_chunk(const int32_t* __restrict__ ids, int T, int E, int k, int tpc, int C,
                                          int* s_wc, Base chunk_base, Off off, int32_t* __restrict__ dest_row,
                                          uint8_t* __restrict__ drop_mask, int32_t* __restrict__ src_token,
                                          int32_t* __restrict__ src_slot) {
    for (int i = threadIdx.x; i < 32 * E; i += blockDim.x) s_wc[i] = 0;
    __syncthreads();
    const int a = threadIdx.x, lane = a & 31, warp = a >> 5;
    const int t = blockIdx.x * tpc + a / k, j = a % k;
    const bool valid = a < tpc * k && t < T;
    const size_t ga = (size_t)blockIdx.x * tpc * k + a;
    int e = valid ? ids[ga] : -1;
    if (e >= E) e = -1;                          // out-of-range id: treated as dropped (flagged by count)
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int intra = __popc(peers & ((1u << lane) - 1u));
    if (e >= 0 && lane == __ffs(peers) - 1) s_wc[warp * E + e] = __popc(peers);
    __syncthreads();
    for (int x = threadIdx.x; x < E; x += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) { int v = s_wc[w * E + x]; s_wc[w * E + x] = run; run += v; }
    }
    __syncthreads();
    if (valid) {
        int d = -1;
        if (e >= 0) {
            const int slot = chunk_base(e) + s_wc[warp * E + e] + intra;
            if (C == 0 || slot < C) {
                d = off(e) + slot;
                src_token[d] = t;
                src_slot[d] = j;
            }
        }
        dest_row[ga] = d;
        drop_mask[ga] = d < 0 ? 1 : 0;
        return d;
    }
    return -1;
}

__global__ void __launch_bounds__(kChunkA)
dispatch_scatter_kernel(const int32_t* __restrict__ ids, int T, int E, int k, int C,
                        const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
                        int32_t* __restrict__ dest_row, uint8_t* __restrict__ drop_mask,
                        int32_t* __restrict__ src_token, int32_t* __restrict__ src_slot) {
    extern __shared__ int s_wc[];
    rank_chunk(ids, T, E, k, kChunkA / k, C, s_wc, [&](int e) { return chunk_base[(size_t)blockIdx.x * E + e]; },
               [&](int e) { return offsets[e]; }, dest_row, drop_mask, src_token, src_slot);
}

// One token's FP8 payload, one warp: lanes 0-15 and 16-31 take alternate blocks of 128 columns (8 columns a
// lane); per block amax over the 16 lanes, scale = amax / 448 (1 for an all-zero block), codes =
// e4m3(x / scale) to nearest even, saturating; codes and (first lane of the half) the scale go to every kept
// destination row dj[j] >= 0, j < k.
__device__ __forceinline__ void fp8_copy_token(const __nv_bfloat16* __restrict__ src, const int (&dj)[16], int k, int h,
                                               uint8_t* __restrict__ buf8, float* __restrict__ scales, int lane) {
    const int half = lane >> 4, hl = lane & 15;
    const int nblk = h / 128;
    constexpr int U = 2;                          // 2 x 2 blocks of 128 columns per iteration
    for (int b0 = 0; b0 < nblk; b0 += 2 * U) {
        Vec16<__nv_bfloat16> v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + 2 * u + half;
            if (b < nblk) v[u] = ld16_stream(src + (size_t)b * 128 + hl * 8);
            else v[u].v = make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int b = b0 + 2 * u + half;
            float f[8];
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[i] = v[u].get(i);
                amax = fmaxf(amax, fabsf(f[i]));
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
            const float sc = amax > 0.f ? amax / 448.f : 1.f;
            uint32_t w[2];
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i] / sc, f[4 * i + 1] / sc),
                                                                         __NV_SATFINITE, __NV_E4M3);
                const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(f[4 * i + 2] / sc,
                                                                                     f[4 * i + 3] / sc),
                                                                         __NV_SATFINITE, __NV_E4M3);
                w[i] = (uint32_t)lo | ((uint32_t)hi << 16);
            }
            if (b < nblk) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (j < k && dj[j] >= 0) {
                        *reinterpret_cast<uint2*>(buf8 + (size_t)dj[j] * h + (size_t)b * 128 + hl * 8) =
                            make_uint2(w[0], w[1]);
                        if (hl == 0) scales[(size_t)dj[j] * nblk + b] = sc;
                    }
            }
        }
    }
}

// Scan, scatter and payload copy in one launch, for small count tables (at most kFusedScanEntries
// entries, chunks of tpc tokens): every block adds up the count table itself (its own chunk base and the
// per-expert totals, in a fixed order) and derives the same offsets; block 0 also publishes offsets, kept
// counts, the rank layout and the tile schedule. Each block then ranks its chunk, copies its tokens' rows
// (one warp per token, x read once) and, in capacity mode, fills its share of the pad rows.
constexpr int kFusedScanEntries = 1 << 15;

// Shared-memory layout of dispatch_fused_kernel, in ints: s_wc [32 E], s_base [E], s_kept [E],
// s_off [E + 1], s_tp [E + 1], s_dest [kChunkA], s_red [2 kChunkA]. The kernel's pointers and the launch's
// allocation both come from here.
__host__ __device__ constexpr int fused_wc(int) { return 0; }
__host__ __device__ constexpr int fused_base(int E) { return 32 * E; }
__host__ __device__ constexpr int fused_kept(int E) { return fused_base(E) + E; }
__host__ __device__ constexpr int fused_off(int E) { return fused_kept(E) + E; }
__host__ __device__ constexpr int fused_tp(int E) { return fused_off(E) + E + 1; }
__host__ __device__ constexpr int fused_dest(int E) { return fused_tp(E) + E + 1; }
__host__ __device__ constexpr int fused_red(int E) { return fused_dest(E) + kChunkA; }          // 2 x kChunkA
__host__ __device__ constexpr int fused_smem_ints(int E) { return fused_red(E) + 2 * kChunkA; }
// Then (bf16 / fp32 payload) the ring of the bulk row copy: kRingMaxStages mbarriers, and the stages from the
// next 128-byte boundary of the shared window (the launch allocates 128 bytes of slack for that).
constexpr int kRingMaxStages = 32;
constexpr uint32_t kRingStageCap = 16384;     // bytes per stage: a row of up to 16 KB is one piece
__host__ __device__ constexpr int fused_bars_byte(int E) { return (fused_smem_ints(E) * 4 + 7) / 8 * 8; }
__host__ __device__ constexpr int fused_ring_byte(int E) { return fused_bars_byte(E) + 8 * kRingMaxStages; }

// Tokens per chunk of the fused path (0: the count table would be too large; use the three-launch path).
// At most max_chunks chunks (the launch uses one chunk per SM so that every block is resident at once; the
// workspace is sized for the bound of 256) and at most kFusedScanEntries table entries.
constexpr int kFusedMaxChunks = 256;
inline int fused_tokens_per_chunk(int T, int E, int k, int max_chunks) {
    if (T <= 0) return 0;
    const int target = std::max(1, std::min(max_chunks, kFusedScanEntries / E));
    const int tpc = std::max(1, cdiv(T, target));
    return tpc * k <= kChunkA ? tpc : 0;
}

// FP8: the payload goes to buf8 / scales as e4m3 codes with per-128-column scales (fp8_copy_token; T is bf16,
// buf unused); pad rows get codes 0 and scale 0.
template <typename T, bool FP8 = false>
__global__ void __launch_bounds__(kChunkA)
dispatch_fused_kernel(const T* __restrict__ x, const int32_t* __restrict__ ids, int T_, int h, int E, int k, int tpc,
                      int C, int R, const int32_t* __restrict__ chunk_counts, int nchunks, T* __restrict__ buf,
                      int32_t* __restrict__ offsets, int32_t* __restrict__ kept_counts,
                      int32_t* __restrict__ rank_counts, int32_t* __restrict__ rank_offsets,
                      int32_t* __restrict__ sched, int32_t* __restrict__ dest_row, uint8_t* __restrict__ drop_mask,
                      int32_t* __restrict__ src_token, int32_t* __restrict__ src_slot, uint8_t* __restrict__ buf8,
                      float* __restrict__ scales, int ring_stages, uint32_t stage_bytes, long long wait_limit,
                      unsigned* __restrict__ err) {
    extern __shared__ int sm[];
    int* s_wc = sm + fused_wc(E);
    int* s_base = sm + fused_base(E);
    int* s_kept = sm + fused_kept(E);
    int* s_off = sm + fused_off(E);
    int* s_tp = sm + fused_tp(E);
    int* s_dest = sm + fused_dest(E);
    int* s_rb = sm + fused_red(E);
    int* s_rt = s_rb + kChunkA;
    __shared__ int s_tmp[32];
    const int t0 = blockIdx.x * tpc;
    const int ntok = min(tpc, T_ - t0);
    {   // this chunk's token rows are known from the start: have L2 fetch them while the count table is summed
        // and the chunk ranked (16-byte multiples: h % 8 == 0). (Issuing the ring's bulk loads here instead was
        // measured: the copy ended no sooner, the issuing thread reached the count table later.)
        const unsigned row_bytes = (unsigned)(h * sizeof(T));
        for (int i = threadIdx.x; i < ntok; i += blockDim.x)
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                         ::"l"(reinterpret_cast<uint64_t>(x + (size_t)(t0 + i) * h)), "r"(row_bytes) : "memory");
    }
    pdl_wait();                               // the count table (dispatch_count_kernel) is complete from here on
    pdl_trigger();                            // the grouped GEMM may launch; it waits for this kernel to complete
    {   // count table -> this chunk's base and the per-expert totals: S slices of chunks per expert in
        // parallel, then a tree over the slices (S = largest power of two with S * E <= kChunkA)
        int S = 1;
        while (S * 2 * E <= kChunkA) S *= 2;
        const int tid = threadIdx.x, sl = tid / E, ex = tid - sl * E;
        if (sl < S) {
            int pb = 0, pt = 0;
            for (int c = sl; c < nchunks; c += 4 * S) {   // up to four loads in flight, the last round too
                int v[4];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    v[u] = c + u * S < nchunks ? __ldg(chunk_counts + (size_t)(c + u * S) * E + ex) : 0;
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    pt += v[u];
                    pb += c + u * S < (int)blockIdx.x ? v[u] : 0;
                }
            }
            s_rb[tid] = pb;
            s_rt[tid] = pt;
        }
        for (int st = S / 2; st > 0; st >>= 1) {
            __syncthreads();
            if (sl < st) { s_rb[tid] += s_rb[tid + st * E]; s_rt[tid] += s_rt[tid + st * E]; }
        }
        __syncthreads();
    }
    const int e = threadIdx.x;
    int total = 0;
    if (e < E) { s_base[e] = s_rb[e]; total = s_rt[e]; }
    layout_from_counts(total, E, C, s_tmp, s_kept, s_off, s_tp);
    if (blockIdx.x == 0)
        publish_layout(E, R, s_kept, s_off, s_tp, offsets, kept_counts, rank_counts, rank_offsets, sched);
    const int d = rank_chunk(ids, T_, E, k, tpc, C, s_wc, [&](int ee) { return s_base[ee]; },
                             [&](int ee) { return s_off[ee]; }, dest_row, drop_mask, src_token, src_slot);
    s_dest[threadIdx.x] = d;
    __syncthreads();

    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if constexpr (FP8) {
        for (int tl = warp; tl < ntok; tl += kChunkA / 32) {
            int dj[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) dj[j] = j < k ? s_dest[tl * k + j] : -1;
            fp8_copy_token(x + (size_t)(t0 + tl) * h, dj, k, h, buf8, scales, lane);
        }
    } else if (threadIdx.x == 0 && ntok > 0) {
        // the rows move through the bulk-copy unit, issued by this one thread; the other warps fill pad rows
        RingCursor rc = ring_start(reinterpret_cast<const char*>(x + (size_t)t0 * h), (uint32_t)(h * sizeof(T)), ntok,
                                   (shared_u32(sm) + (uint32_t)fused_ring_byte(E) + 127u) & ~127u,
                                   shared_u32(sm) + (uint32_t)fused_bars_byte(E), ring_stages, stage_bytes);
        ring_finish(rc, k, s_dest, reinterpret_cast<char*>(buf), wait_limit, err);
    }
    if (C > 0) {
        // Pad rows, numbered in expert order (q = pads of earlier experts + p), are spread evenly over the blocks
        // and then over each block's fill warps (all warps with the FP8 payload, warps 1-31 otherwise): row q goes
        // to fill warp (q mod grid) * FW + (q / grid) mod FW, so that every block fills about the same number.
        constexpr int FW = FP8 ? kChunkA / 32 : kChunkA / 32 - 1;
        if (!FP8 && warp == 0) return;
        const int G = gridDim.x, b = blockIdx.x, fw = FP8 ? warp : warp - 1;
        const long long step = (long long)G * FW;
        long long run = 0;                                // pads of earlier experts = rq * G + rr
        int rq = 0, rr = 0;
        for (int ee = 0; ee < E; ++ee) {
            const int npad = C - s_kept[ee];
            // this warp's first pad row q >= run: q mod G == b (the first such row is in column a = q / G), then
            // the first of a, a + 1, ... congruent to fw mod FW; after it every G * FW rows
            const int a = rq + (b < rr ? 1 : 0);
            const long long q1 = ((long long)a + ((fw - a % FW) % FW + FW) % FW) * G + b;
            for (long long q = q1; q - run < npad; q += step) {
                const long long r = (long long)ee * C + s_kept[ee] + (q - run);
                if (lane == 0) { src_token[r] = -1; src_slot[r] = -1; }
                if constexpr (FP8) {
                    for (int d0 = lane * 16; d0 < h; d0 += 32 * 16)
                        *reinterpret_cast<uint4*>(buf8 + r * h + d0) = make_uint4(0, 0, 0, 0);
                    for (int sb = lane; sb < h / 128; sb += 32) scales[r * (h / 128) + sb] = 0.f;
                } else {
                    Vec16<T> z;
                    z.v = {};
                    for (int d0 = lane * V; d0 < h; d0 += 32 * V) st16(buf + r * h + d0, z);
                }
            }
            run += npad;
            rq += npad / G;
            rr += npad % G;
            if (rr >= G) { rr -= G; ++rq; }
        }
    }
}

// Blocks [0, tok_blocks): one warp per token, read x[t] once and write it to each kept destination row.
// Blocks [tok_blocks, grid) (capacity mode): pad rows [offsets[e] + kept[e], offsets[e + 1]) get a zero
// payload and src = -1.
template <typename T>
__global__ void __launch_bounds__(256)
dispatch_copy_pad_kernel(const T* __restrict__ x, const int32_t* __restrict__ dest_row, int T_, int h, int k,
                         T* __restrict__ buf, int tok_blocks, const int32_t* __restrict__ kept_counts, int E, int C,
                         int32_t* __restrict__ src_token, int32_t* __restrict__ src_slot) {
    constexpr int V = Vec16<T>::N;
    const int lane = threadIdx.x & 31;
    if ((int)blockIdx.x < tok_blocks) {
        const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
        if (t >= T_) return;
        const int my = lane < k ? dest_row[(size_t)t * k + lane] : -1;
        int dj[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) dj[j] = __shfl_sync(0xffffffffu, my, j);   // all lanes, before any exit
        const T* src = x + (size_t)t * h;
        constexpr int U = 4;                      // 16-byte loads in flight per lane
        for (int d0 = lane * V; d0 < h; d0 += U * 32 * V) {
            Vec16<T> v[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (d0 + u * 32 * V < h) v[u] = ld16_stream(src + d0 + u * 32 * V);
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < k && dj[j] >= 0) {
#pragma unroll
                    for (int u = 0; u < U; ++u)
                        if (d0 + u * 32 * V < h) st16(buf + (size_t)dj[j] * h + d0 + u * 32 * V, v[u]);
                }
        }
        return;
    }
    const long long rows = (long long)E * C;
    const int nb = gridDim.x - tok_blocks;
    for (long long r = (long long)(blockIdx.x - tok_blocks) * 8 + (threadIdx.x >> 5); r < rows; r += (long long)nb * 8) {
        const int e = (int)(r / C);
        if (r - (long long)e * C < kept_counts[e]) continue;
        if (lane == 0) { src_token[r] = -1; src_slot[r] = -1; }
        Vec16<T> z;
        z.v = {};
        for (int d0 = lane * V; d0 < h; d0 += 32 * V) st16(buf + r * h + d0, z);
    }
}

// FP8 send buffer ("10.5 序列并行与专家并行", section 10.5.7: activations cross nodes in a low-precision
// format such as FP8, halving the bytes). Blocks [0, tok_blocks): one warp per token, quantised once: each
// half-warp covers one 128-column block with 8 columns per lane; amax over the half-warp, s = amax / 448 (1 for
// an all-zero block), codes = e4m3(x / s) rounded to nearest even with saturation; the 8 code bytes of a lane
// and (first lane of the half) the scale go to every kept destination row. Blocks [tok_blocks, grid): pad rows
// (capacity mode) get codes 0, scale 0 and src = -1.
__global__ void __launch_bounds__(256)
dispatch_copy_fp8_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ dest_row, int T_, int h,
                         int k, uint8_t* __restrict__ buf8, float* __restrict__ scales, int tok_blocks,
                         const int32_t* __restrict__ kept_counts, int E, int C, int32_t* __restrict__ src_token,
                         int32_t* __restrict__ src_slot) {
    const int lane = threadIdx.x & 31;
    const int nblk = h / 128;
    if ((int)blockIdx.x < tok_blocks) {
        const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
        if (t >= T_) return;
        const int my = lane < k ? dest_row[(size_t)t * k + lane] : -1;
        int dj[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) dj[j] = __shfl_sync(0xffffffffu, my, j);
        fp8_copy_token(x + (size_t)t * h, dj, k, h, buf8, scales, lane);
        return;
    }
    const long long rows = (long long)E * C;
    const int nb = gridDim.x - tok_blocks;
    for (long long r = (long long)(blockIdx.x - tok_blocks) * 8 + (threadIdx.x >> 5); r < rows; r += (long long)nb * 8) {
        const int e = (int)(r / C);
        if (r - (long long)e * C < kept_counts[e]) continue;
        if (lane == 0) { src_token[r] = -1; src_slot[r] = -1; }
        for (int d0 = lane * 16; d0 < h; d0 += 32 * 16)
            *reinterpret_cast<uint4*>(buf8 + r * h + d0) = make_uint4(0, 0, 0, 0);
        for (int b = lane; b < nblk; b += 32) scales[r * nblk + b] = 0.f;
    }
}

__global__ void dense_sched_kernel(int rows, int32_t* sched) {
    const int ntiles = (rows + MOE_TILE_M - 1) / MOE_TILE_M;
    if (blockIdx.x == 0 && threadIdx.x == 0) { sched[0] = ntiles; sched[1] = 1; sched[2] = 0; sched[3] = ntiles; }
    int4* tiles = reinterpret_cast<int4*>(sched + sched_tiles_offset(1));
    for (int m = blockIdx.x * blockDim.x + threadIdx.x; m < ntiles; m += gridDim.x * blockDim.x)
        tiles[m] = make_int4(0, m * MOE_TILE_M, min(rows, (m + 1) * MOE_TILE_M), 0);
}

static int num_chunks(int T, int k) { return T <= 0 ? 0 : cdiv(T, kChunkA / k); }
// Threads of a count block: one per assignment of its chunk, in whole warps (a chunk of the fused path holds
// far fewer than kChunkA assignments when T is small next to the SM count: 54 at the page-3 shape).
static int count_threads(int tpc, int k) { return std::max(32, std::min(kChunkA, (tpc * k + 31) / 32 * 32)); }

// Ring of the fused kernel's bulk row copy: stages of min(row bytes, 16 KB), as many as fit (at most 32)
// beside the kernel's tables in 227 KB of shared memory less 1 KB for its static variables and margin.
struct RingPlan { int stages; uint32_t stage_bytes; size_t smem; };
static RingPlan ring_plan(int E, size_t row_bytes) {
    constexpr size_t kSmemMax = 227 * 1024 - 1024;
    RingPlan r;
    r.stage_bytes = (uint32_t)std::min<size_t>(row_bytes, kRingStageCap);
    const size_t base = (size_t)fused_ring_byte(E) + 128;
    r.stages = (int)std::min<size_t>(kRingMaxStages, base < kSmemMax ? (kSmemMax - base) / r.stage_bytes : 0);
    r.smem = base + (size_t)r.stages * r.stage_bytes;
    return r;
}
static int num_fused_chunks(int T, int E, int k) {
    const int tpc = fused_tokens_per_chunk(T, E, k, kFusedMaxChunks);
    return tpc ? cdiv(T, tpc) : 0;
}

}  // namespace moe

using namespace moe;

extern "C" size_t moe_dispatch_rows(int T, int E, int k, int capacity) {
    if (T < 0 || E <= 0 || k <= 0) return 0;
    return capacity > 0 ? (size_t)E * capacity : (size_t)T * k;
}

extern "C" size_t moe_tile_sched_bytes(int T, int E, int k, int capacity) {
    if (T < 0 || E <= 0 || k <= 0) return 0;
    return sched_words((long long)moe_dispatch_rows(T, E, k, capacity), E) * sizeof(int32_t);
}

extern "C" size_t moe_dispatch_workspace_size(int T, int E, int k, int capacity) {
    (void)capacity;
    if (T < 0 || E <= 0 || k <= 0 || k > kChunkA) return 0;
    const int nch = std::max(num_chunks(T, k), num_fused_chunks(T, E, k));
    return align_up((size_t)nch * E * sizeof(int32_t), 256);
}

extern "C" int moe_dispatch(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity,
                            int num_ranks, int dtype, void* buf, int32_t* offsets, int32_t* kept_counts,
                            int32_t* dest_row, uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot,
                            int32_t* rank_counts, int32_t* rank_offsets, int32_t* tile_sched, void* ws,
                            size_t ws_bytes, void* stream) {
    MOE_REQUIRE(dtype == MOE_F32 || dtype == MOE_BF16, MOE_ERR_UNSUPPORTED, "moe_dispatch: dtype %d", dtype);
    MOE_REQUIRE(T >= 0 && h > 0 && h % 8 == 0, MOE_ERR_INVALID_ARG, "moe_dispatch: T=%d h=%d", T, h);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 16, MOE_ERR_INVALID_ARG,
                "moe_dispatch: E=%d k=%d", E, k);
    MOE_REQUIRE(capacity >= 0, MOE_ERR_INVALID_ARG, "moe_dispatch: capacity %d < 0", capacity);
    MOE_REQUIRE(num_ranks >= 1 && num_ranks <= E && E % num_ranks == 0, MOE_ERR_INVALID_ARG,
                "moe_dispatch: num_ranks %d must divide E=%d", num_ranks, E);
    const long long rows = (long long)moe_dispatch_rows(T, E, k, capacity);
    MOE_REQUIRE(rows < (1LL << 31), MOE_ERR_INVALID_ARG, "moe_dispatch: %lld rows overflow int32", rows);
    MOE_REQUIRE(offsets && kept_counts && rank_counts && rank_offsets && tile_sched, MOE_ERR_INVALID_ARG,
                "moe_dispatch: null pointer");
    MOE_REQUIRE(T == 0 || (x && topk_ids && dest_row && drop_mask), MOE_ERR_INVALID_ARG, "moe_dispatch: null pointer");
    MOE_REQUIRE(rows == 0 || (buf && src_token && src_slot), MOE_ERR_INVALID_ARG, "moe_dispatch: null pointer");
    MOE_REQUIRE(aligned16(x) && aligned16(buf) && aligned16(tile_sched), MOE_ERR_INVALID_ARG,
                "moe_dispatch: x, buf and tile_sched must be 16-byte aligned");
    const size_t need = moe_dispatch_workspace_size(T, E, k, capacity);
    MOE_REQUIRE(ws_bytes >= need && (need == 0 || ws), MOE_ERR_WORKSPACE, "moe_dispatch: workspace %zu < %zu",
                ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "moe_dispatch: device error word unavailable");
    int32_t* chunk = static_cast<int32_t*>(ws);
    const int tpc_f = fused_tokens_per_chunk(T, E, k, std::min(kFusedMaxChunks, num_sms()));
    if (tpc_f > 0) {
        const int nch = cdiv(T, tpc_f);
        dispatch_count_kernel<<<nch, count_threads(tpc_f, k), E * sizeof(int), s>>>(topk_ids, T, E, k, tpc_f, chunk, err);
        if (int rc = check_launch("dispatch_count_kernel")) return rc;
        const RingPlan rp = ring_plan(E, (size_t)h * (dtype == MOE_BF16 ? 2 : 4));
        MOE_REQUIRE(rp.stages >= 2, MOE_ERR_INVALID_ARG, "moe_dispatch: no room for the copy ring (E=%d, h=%d)", E, h);
        const size_t smem = rp.smem;
        const long long wl = wait_limit();
        cudaError_t le;
        if (dtype == MOE_BF16) {
            cudaFuncSetAttribute(dispatch_fused_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
            le = launch_pdl(dispatch_fused_kernel<__nv_bfloat16>, dim3(nch), dim3(kChunkA), smem, s,
                static_cast<const __nv_bfloat16*>(x), topk_ids, T, h, E, k, tpc_f, capacity, num_ranks,
                (const int32_t*)chunk, nch, static_cast<__nv_bfloat16*>(buf), offsets, kept_counts, rank_counts,
                rank_offsets, tile_sched, dest_row, drop_mask, src_token, src_slot, (uint8_t*)nullptr, (float*)nullptr,
                rp.stages, rp.stage_bytes, wl, err);
        } else {
            cudaFuncSetAttribute(dispatch_fused_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            le = launch_pdl(dispatch_fused_kernel<float>, dim3(nch), dim3(kChunkA), smem, s, static_cast<const float*>(x),
                topk_ids, T, h, E, k, tpc_f, capacity, num_ranks, (const int32_t*)chunk, nch, static_cast<float*>(buf),
                offsets, kept_counts, rank_counts, rank_offsets, tile_sched, dest_row, drop_mask, src_token, src_slot,
                (uint8_t*)nullptr, (float*)nullptr, rp.stages, rp.stage_bytes, wl, err);
        }
        return check_launch(le, "dispatch_fused_kernel");
    }
    // large count tables (or no tokens): count, scan, scatter, then copy and pad fill
    const int nch = num_chunks(T, k);
    if (nch > 0) {
        dispatch_count_kernel<<<nch, kChunkA, E * sizeof(int), s>>>(topk_ids, T, E, k, kChunkA / k, chunk, err);
        if (int rc = check_launch("dispatch_count_kernel")) return rc;
    }
    dispatch_scan_kernel<<<1, 1024, 0, s>>>(chunk, nch, E, capacity, num_ranks, offsets, kept_counts, rank_counts,
                                           rank_offsets, tile_sched);
    if (int rc = check_launch("dispatch_scan_kernel")) return rc;
    if (nch > 0) {
        const size_t smem = (size_t)32 * E * sizeof(int);
        cudaFuncSetAttribute(dispatch_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        dispatch_scatter_kernel<<<nch, kChunkA, smem, s>>>(topk_ids, T, E, k, capacity, chunk, offsets, dest_row,
                                                          drop_mask, src_token, src_slot);
        if (int rc = check_launch("dispatch_scatter_kernel")) return rc;
    }
    const int tok_blocks = cdiv(T, 8);
    const int pad_blocks = (capacity > 0 && rows > 0) ? std::min(cdiv(rows, 8), 2 * num_sms()) : 0;
    if (tok_blocks + pad_blocks > 0) {
        if (dtype == MOE_BF16)
            dispatch_copy_pad_kernel<__nv_bfloat16><<<tok_blocks + pad_blocks, 256, 0, s>>>(
                static_cast<const __nv_bfloat16*>(x), dest_row, T, h, k, static_cast<__nv_bfloat16*>(buf), tok_blocks,
                kept_counts, E, capacity, src_token, src_slot);
        else
            dispatch_copy_pad_kernel<float><<<tok_blocks + pad_blocks, 256, 0, s>>>(
                static_cast<const float*>(x), dest_row, T, h, k, static_cast<float*>(buf), tok_blocks, kept_counts, E,
                capacity, src_token, src_slot);
        if (int rc = check_launch("dispatch_copy_pad_kernel")) return rc;
    }
    return MOE_OK;
}

namespace moe {
int launch_dense_sched(int rows, int32_t* sched, cudaStream_t s) {
    const int ntiles = cdiv(rows, MOE_TILE_M);
    dense_sched_kernel<<<std::max(1, std::min(cdiv(ntiles, 256), 64)), 256, 0, s>>>(rows, sched);
    return check_launch("dense_sched_kernel");
}
}  // namespace moe

extern "C" int moe_dense_tile_sched(int rows, int32_t* tile_sched, void* stream) {
    MOE_REQUIRE(rows >= 0 && tile_sched && aligned16(tile_sched), MOE_ERR_INVALID_ARG,
                "moe_dense_tile_sched: rows=%d, tile_sched must be non-null and 16-byte aligned", rows);
    return launch_dense_sched(rows, tile_sched, static_cast<cudaStream_t>(stream));
}


// ---------------------------------------------------------------------------------------------------
// moe_dispatch_static: the same dispatch for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc, or any allocator, at the point where they dispatch tokens: code that
// runs inside a host framework which owns all device memory and hands plugins only the tensors of a call,
// real-time or latency-critical threads where an allocation (and the device synchronisation it may imply)
// is not allowed, and programs that must reserve every byte of device memory once at start-up. For them
// this entry point keeps its scratch (the per-chunk expert counts) in a fixed array in the library's own
// device memory instead of a caller-provided workspace; the caller still passes every input and output.
//
// The array is a file-scope __device__ variable: every GPU that loads the library holds it until the process
// exits. Its host-side name is only a stand-in for the symbol, never a device address, so the first call on
// each device, with that device current, looks its address up with cudaGetSymbolAddress and caches it; make
// that first call on a device before capturing a stream on it. The cache remembers the context it was filled in
// and a call in another context (after cudaDeviceReset, say) looks the address up again, so make the first
// call after a reset before any capture as well. All calls share the one array: calls whose
// kernels may overlap on the GPU (different streams, no ordering between them) race on it and must be
// serialised by the caller. Nothing in the array has to start at zero: every call writes each word before it
// reads it, so the contents left by the previous call do not matter.
// ---------------------------------------------------------------------------------------------------
namespace moe {
constexpr size_t kStaticScratchBytes = (size_t)1 << 20;     // 1 MiB: ceil(T / (1024/k)) chunks x E x 4 B
static __device__ __align__(256) int32_t g_dispatch_scratch[kStaticScratchBytes / sizeof(int32_t)];
static std::mutex g_static_mu;
static void* g_static_ptr[64];
static unsigned long long g_static_ctx[64];     // the context the address was looked up in, per device
}  // namespace moe

extern "C" int moe_dispatch_static(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity,
                                   int num_ranks, int dtype, void* buf, int32_t* offsets, int32_t* kept_counts,
                                   int32_t* dest_row, uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot,
                                   int32_t* rank_counts, int32_t* rank_offsets, int32_t* tile_sched, void* stream) {
    MOE_REQUIRE(T >= 0 && E >= 1 && E <= 1024 && k >= 1 && k <= 16, MOE_ERR_INVALID_ARG,
                "moe_dispatch_static: T=%d E=%d k=%d", T, E, k);
    const size_t need = moe_dispatch_workspace_size(T, E, k, capacity);
    MOE_REQUIRE(need <= moe::kStaticScratchBytes, MOE_ERR_INVALID_ARG,
                "moe_dispatch_static: T=%d, E=%d, k=%d needs %zu scratch bytes, more than the static %zu; "
                "use moe_dispatch with a workspace instead", T, E, k, need, moe::kStaticScratchBytes);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    MOE_REQUIRE(e == cudaSuccess && dev >= 0 && dev < 64, MOE_ERR_CUDA, "moe_dispatch_static: no current device (%s)",
                cudaGetErrorString(e));
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(moe::g_static_mu);
        const unsigned long long ctx = moe::context_id();
        if (!moe::g_static_ptr[dev] || ctx == 0 || moe::g_static_ctx[dev] != ctx) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, moe::g_dispatch_scratch);
            MOE_REQUIRE(e == cudaSuccess && p, MOE_ERR_CUDA, "moe_dispatch_static: cudaGetSymbolAddress failed: %s",
                        cudaGetErrorString(e));
            moe::g_static_ptr[dev] = p;
            moe::g_static_ctx[dev] = moe::context_id();
        }
        scratch = moe::g_static_ptr[dev];
    }
    return moe_dispatch(x, topk_ids, T, h, E, k, capacity, num_ranks, dtype, buf, offsets, kept_counts, dest_row,
                        drop_mask, src_token, src_slot, rank_counts, rank_offsets, tile_sched, scratch,
                        moe::kStaticScratchBytes, stream);
}

namespace moe {
// out [rows, h] bf16 = bf16(fp32(e4m3 value of buf8[r, c]) * scales[r, c / 128]): 16 codes per thread pass.
__global__ void __launch_bounds__(256)
dequant_fp8_kernel(const uint8_t* __restrict__ buf8, const float* __restrict__ scales, long long rows, int h,
                   __nv_bfloat16* __restrict__ out) {
    const int vpr = h / 16, nb = h / 128;
    const long long n = rows * vpr;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const long long r = i / vpr;
        const int c = (int)(i - r * vpr) * 16;
        const float sc = __ldg(scales + r * nb + (c >> 7));
        const uint4 q = __ldcs(reinterpret_cast<const uint4*>(buf8 + r * h + c));
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int hw = 0; hw < 8; ++hw) {
            const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((qw[hw >> 1] >> (16 * (hw & 1))) & 0xFFFFu);
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
            const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            const __nv_bfloat162 bv = __floats2bfloat162_rn(fv.x * sc, fv.y * sc);
            o[hw] = *reinterpret_cast<const uint32_t*>(&bv);
        }
        uint4* dst = reinterpret_cast<uint4*>(out + r * h + c);
        dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}
}  // namespace moe

extern "C" int moe_dequant_fp8(const uint8_t* buf8, const float* scales, int rows, int h, void* out, void* stream) {
    MOE_REQUIRE(rows >= 0 && h > 0 && h % 128 == 0, MOE_ERR_INVALID_ARG, "moe_dequant_fp8: rows=%d h=%d (need h%%128==0)",
                rows, h);
    if (rows == 0) return MOE_OK;
    MOE_REQUIRE(buf8 && scales && out, MOE_ERR_INVALID_ARG, "moe_dequant_fp8: null pointer");
    MOE_REQUIRE(aligned16(buf8) && aligned16(out), MOE_ERR_INVALID_ARG,
                "moe_dequant_fp8: buf8 and out must be 16-byte aligned");
    const long long n = (long long)rows * (h / 16);
    const int grid = (int)std::min<long long>(cdiv(n, 256), 8LL * num_sms());
    dequant_fp8_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(buf8, scales, rows, h,
                                                                            static_cast<__nv_bfloat16*>(out));
    return check_launch("dequant_fp8_kernel");
}

extern "C" int moe_dispatch_fp8(const void* x, const int32_t* topk_ids, int T, int h, int E, int k, int capacity,
                                int num_ranks, uint8_t* buf8, float* scales, int32_t* offsets, int32_t* kept_counts,
                                int32_t* dest_row, uint8_t* drop_mask, int32_t* src_token, int32_t* src_slot,
                                int32_t* rank_counts, int32_t* rank_offsets, int32_t* tile_sched, void* ws,
                                size_t ws_bytes, void* stream) {
    MOE_REQUIRE(T >= 0 && h > 0 && h % 128 == 0, MOE_ERR_INVALID_ARG, "moe_dispatch_fp8: T=%d h=%d (need h%%128==0)",
                T, h);
    MOE_REQUIRE(E >= 1 && E <= 1024 && k >= 1 && k <= E && k <= 16, MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: E=%d k=%d", E, k);
    MOE_REQUIRE(capacity >= 0, MOE_ERR_INVALID_ARG, "moe_dispatch_fp8: capacity %d < 0", capacity);
    MOE_REQUIRE(num_ranks >= 1 && num_ranks <= E && E % num_ranks == 0, MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: num_ranks %d must divide E=%d", num_ranks, E);
    const long long rows = (long long)moe_dispatch_rows(T, E, k, capacity);
    MOE_REQUIRE(rows < (1LL << 31), MOE_ERR_INVALID_ARG, "moe_dispatch_fp8: %lld rows overflow int32", rows);
    MOE_REQUIRE(offsets && kept_counts && rank_counts && rank_offsets && tile_sched, MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: null pointer");
    MOE_REQUIRE(T == 0 || (x && topk_ids && dest_row && drop_mask), MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: null pointer");
    MOE_REQUIRE(rows == 0 || (buf8 && scales && src_token && src_slot), MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: null pointer");
    MOE_REQUIRE(aligned16(x) && aligned16(buf8) && aligned16(tile_sched), MOE_ERR_INVALID_ARG,
                "moe_dispatch_fp8: x, buf8 and tile_sched must be 16-byte aligned");
    const size_t need = moe_dispatch_workspace_size(T, E, k, capacity);
    MOE_REQUIRE(ws_bytes >= need && (need == 0 || ws), MOE_ERR_WORKSPACE, "moe_dispatch_fp8: workspace %zu < %zu",
                ws_bytes, need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "moe_dispatch_fp8: device error word unavailable");
    int32_t* chunk = static_cast<int32_t*>(ws);
    const int tpc_f = fused_tokens_per_chunk(T, E, k, std::min(kFusedMaxChunks, num_sms()));
    if (tpc_f > 0) {                              // count, then scan + scatter + quantised copy in one launch
        const int nchf = cdiv(T, tpc_f);
        dispatch_count_kernel<<<nchf, count_threads(tpc_f, k), E * sizeof(int), s>>>(topk_ids, T, E, k, tpc_f, chunk,
                                                                                   err);
        if (int rc = check_launch("dispatch_count_kernel")) return rc;
        const size_t smem = (size_t)fused_smem_ints(E) * sizeof(int);
        cudaFuncSetAttribute(dispatch_fused_kernel<__nv_bfloat16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
        const cudaError_t le = launch_pdl(dispatch_fused_kernel<__nv_bfloat16, true>, dim3(nchf), dim3(kChunkA), smem, s,
            static_cast<const __nv_bfloat16*>(x), topk_ids, T, h, E, k, tpc_f, capacity, num_ranks, (const int32_t*)chunk,
            nchf, (__nv_bfloat16*)nullptr, offsets, kept_counts, rank_counts, rank_offsets, tile_sched, dest_row,
            drop_mask, src_token, src_slot, buf8, scales, 0, 0u, 0LL, err);
        return check_launch(le, "dispatch_fused_kernel<fp8>");
    }
    const int nch = num_chunks(T, k);
    if (nch > 0) {
        dispatch_count_kernel<<<nch, kChunkA, E * sizeof(int), s>>>(topk_ids, T, E, k, kChunkA / k, chunk, err);
        if (int rc = check_launch("dispatch_count_kernel")) return rc;
    }
    dispatch_scan_kernel<<<1, 1024, 0, s>>>(chunk, nch, E, capacity, num_ranks, offsets, kept_counts, rank_counts,
                                           rank_offsets, tile_sched);
    if (int rc = check_launch("dispatch_scan_kernel")) return rc;
    if (nch > 0) {
        const size_t smem = (size_t)32 * E * sizeof(int);
        cudaFuncSetAttribute(dispatch_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        dispatch_scatter_kernel<<<nch, kChunkA, smem, s>>>(topk_ids, T, E, k, capacity, chunk, offsets, dest_row,
                                                          drop_mask, src_token, src_slot);
        if (int rc = check_launch("dispatch_scatter_kernel")) return rc;
    }
    const int tok_blocks = cdiv(T, 8);
    const int pad_blocks = (capacity > 0 && rows > 0) ? std::min(cdiv(rows, 8), 2 * num_sms()) : 0;
    if (tok_blocks + pad_blocks > 0) {
        dispatch_copy_fp8_kernel<<<tok_blocks + pad_blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), dest_row,
            T, h, k, buf8, scales, tok_blocks, kept_counts, E, capacity, src_token, src_slot);
        if (int rc = check_launch("dispatch_copy_fp8_kernel")) return rc;
    }
    return MOE_OK;
}
