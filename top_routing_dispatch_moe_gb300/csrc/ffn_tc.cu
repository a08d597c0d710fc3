// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05, sm_103a), bf16 operands with
// fp32 accumulation in tensor memory.
//
// "Megatron-LM 分布式训练（六）", data flow: the local experts run as one GroupedGEMM; "v6 长序列和 MoE",
// table row "expert" (each expert's FFN h -> F -> h) and the follow-up note (sort tokens by expert, one
// grouped GEMM instead of E small launches).
//
// One persistent kernel per GEMM, one CTA per SM, 6 warps with fixed roles:
//   warp 0  TMA producer: 128x64 A tiles (token rows of one expert) and 256x64 B tiles (weight rows) into a
//           4-stage shared-memory ring, 128-byte swizzled, completion counted on one mbarrier per stage;
//   warp 1  allocates all 512 tensor-memory columns (two 128x256 fp32 accumulators) and issues the
//           tcgen05.mma (M=128, N=256, K=16) from one thread; tcgen05.commit frees a stage once the MMAs
//           that read it are done and signals a full accumulator after the last K step;
//   warps 2-5  epilogue: tcgen05.ld of the accumulator rows (one TMEM lane = one output row per thread),
//           then either silu(gate) * up -> bf16 act (up/gate GEMM; the packed B tile holds 128 gate and the
//           matching 128 up rows) or a plain bf16 conversion (down GEMM), masked to the expert's rows.
// The two accumulators let the epilogue of tile i overlap the MMAs of tile i+1.
//
// Work items are (m-tile, n-tile) pairs over the device tile schedule written by dispatch, ordered expert by
// expert, n-tile by n-tile, m-tile fastest: CTAs running at the same time share one expert's token rows and
// one 256-row weight tile, so weights are read from HBM about once. Nothing about the routing is known on
// the host: the kernel reads the tile count and per-expert tile prefix from device memory.
//
// Every mbarrier wait is bounded. A wait that runs out latches MOE_ERR_TIMEOUT into the device error word
// and raises a CTA-wide abort flag; every role then leaves its loop, the producer waits (bounded) for its
// TMA copies in flight, the MMA thread waits (bounded) for its MMAs, and the tensor memory is freed before
// the CTA exits.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <cuda_fp8.h>
#include <algorithm>
#include <mutex>
#include "ffn.cuh"

namespace moe {
namespace tc {

constexpr int BM = 128;                      // rows per tile (UMMA M, one TMEM lane per row)
constexpr int BK = 64;                       // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int UK = 16;                       // K per tcgen05.mma (kind::f16)
constexpr int A_BYTES = BM * BK * 2;         // 16 KB
constexpr int TMEM_COLS = 512;               // 2 accumulators x up to 256 fp32 columns
constexpr int NUM_THREADS = 192;
constexpr int NUM_THREADS_A8 = 448;          // + 8 warps that dequantise an e4m3 A operand into the bf16 stage
constexpr int A8_CONVERTER_WARPS = 8;
constexpr int A8_BYTES = BM * BK;            // 8 KB: a 128 x 64 e4m3 tile

// Tile width (UMMA N) and ring depth: 256 columns x 4 stages of 48 KB. (A 192-column tile with 5 stages of
// 40 KB was measured for the down GEMM: 2 % faster on the page-3 shape, where it shortens the last wave,
// 6-17 % slower on the others, which pay for the extra operand bytes per flop.)
template <int BN_, int STAGES_>
struct TileCfg {
    static constexpr int BN = BN_;
    static constexpr int STAGES = STAGES_;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int SMEM_BYTES = 1024 /* alignment slack */ + STAGES * STAGE_BYTES + 256 /* barriers, flags */;
    static constexpr int SMEM_BYTES_A8 = SMEM_BYTES + STAGES * A8_BYTES;   // + the e4m3 staging tiles
    static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "UMMA N for M = 128");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
};
using Wide = TileCfg<256, 4>;
// fp32-output products at most 128 wide (the router logits of up to 128 experts): half the MMA work per tile of
// the 256-wide one, which such a product would fill only half of, and six stages of 32 KB
using Mid = TileCfg<128, 6>;
constexpr long long kDrainLimit = 1LL << 24;

// ---------------------------------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait: true when the phase completed; false when another role aborted or the limit ran out
// (then the abort flag is raised and the timeout latched).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, long long limit, volatile int* abort_flag,
                                           unsigned* err, unsigned site) {
    for (long long i = 0; i < limit; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    *abort_flag = 1;
    latch_device_error(err, kDevErrTimeout, site);
    return false;
}
// Drain wait at exit: no abort check, fixed limit.
__device__ __forceinline__ void drain_phase(uint32_t bar, uint32_t parity, unsigned* err, unsigned site) {
    for (long long i = 0; i < kDrainLimit; ++i)
        if (mbar_try_wait(bar, parity)) return;
    latch_device_error(err, kDevErrTimeout, site);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Tile store shared -> global through the tensor map (rows and columns outside the map's extents are not
// written); bulk-group completion, so the issuing thread waits on its own groups.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4u(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
__device__ __forceinline__ void bulk_wait_read_but1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void st_shared_v4(uint32_t addr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d) : "memory");
}
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, A: M x K (K-major), B: N x K (K-major), bf16 in, fp32 accumulate.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this warp's 32 TMEM lanes (one row per thread).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with 128-byte swizzling: rows of 128
// bytes, 8-row core groups 1024 bytes apart (stride byte offset), leading byte offset unused for this
// layout (set to 16 bytes), descriptor version 1 (bits 46-48), swizzle mode 2 = 128B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);          // start address
    d |= (uint64_t)(16u >> 4) << 16;                     // leading byte offset
    d |= (uint64_t)(1024u >> 4) << 32;                   // stride byte offset
    d |= (uint64_t)1 << 46;                              // version
    d |= (uint64_t)2 << 61;                              // 128B swizzle
    return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits 7-9, 10-12 = 1), both
// K-major (bits 15, 16 = 0), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
template <int N, int M = BM>
__host__ __device__ constexpr uint32_t idesc_bf16() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Epilogues: SwiGLU of the packed gate/up tile -> bf16 act; plain bf16 conversion; fp32 (+ per-column bias),
// used for the router logits and the weight gradients; SwiGLU backward of the packed gate/up tile (reads the
// act gradient, writes the gate and up pre-activation gradients in the packed column order).
// EPI_SWIGLU_SAVE: EPI_SWIGLU that also stores the pre-activations (Params::gu_out / sh_gu_out); a separate
// instantiation, so that the plain forward carries no trace of it.
// EPI_BF16_COMBINE: the plain bf16 epilogue of the down GEMM, after which the tile that completes a token's
// column block also combines it into y (combine_arrive).
enum Epi : int { EPI_SWIGLU = 0, EPI_BF16 = 1, EPI_F32 = 2, EPI_SWIGLU_BWD = 3, EPI_SWIGLU_SAVE = 4, EPI_BF16_COMBINE = 5 };
__host__ __device__ constexpr bool plain_bf16(int epi) { return epi == EPI_BF16 || epi == EPI_BF16_COMBINE; }

struct Params {
    const int32_t* sched;
    int K;              // reduction length
    int NT;             // n-tiles per expert
    int b_rows;         // B rows per expert in the B tensor map (2 Fp for up/gate, h for down, E for the router)
    int n_valid;        // valid output columns (F for up/gate, h for down, E for the router)
    int ldo;            // output leading dimension
    __nv_bfloat16* out;
    float* out_f32;     // EPI_F32 output
    const float* bias;  // EPI_F32: per-column bias or null
    unsigned* err;
    long long wait_limit;
    int sh_rows;              // rows of the shared expert's dense group in the same launch (0: none)
    __nv_bfloat16* sh_out;    // its output ([sh_rows, ldo])
    const __nv_bfloat16* d_act;   // EPI_SWIGLU_BWD: act gradient [rows, n_valid]
    // weight-gradient mapping (wg_E > 0, one-SM kernel): item = (expert e, n-tile, m-tile), A rows m-tile of
    // wg_M rows, B rows n-tile, K = expert e's segment [seg[e], seg[e + 1]) of the transposed operands.
    int wg_E, wg_MT, wg_M;
    const int32_t* seg;
    int wg_gu;                // rows are the packed gate/up order: block b of 128 rows -> out_f32 (gate, b even)
                              // or out2 (up, b odd), row (b / 2) * 128 + i of expert e's [F][ldo] matrix
    int wg_F;                 // wg_gu: valid rows F of each de-interleaved matrix
    float* out2;
    // e4m3 A operand (A8 kernels): value = bf16(fp32(e4m3) * a_scales[row * a_nblk + column / 128]), rows < a_rows
    const float* a_scales;
    int a_nblk, a_rows;
    // weight-gradient mapping without a segment array (seg == null): part e covers columns
    // [e * wg_kchunk, min(K, (e + 1) * wg_kchunk)), wg_kchunk a multiple of BK (split-K partial products)
    int wg_kchunk;
    // one-SM kernel: column extents of the A and B tensor maps (0: K) and the operands' column of reduction
    // index k, k mod kmod (0: k), for a K range that runs over one operand several times (a multiple of BK)
    int a_cols, b_cols, a_kmod, b_kmod;
    // EPI_SWIGLU_SAVE: the pre-activations g and u (bf16) of the routed / shared rows, [rows][NT * 256] in the
    // packed gate/up column order (block n: 128 columns of g, then the u of the same f)
    __nv_bfloat16* gu_out;
    __nv_bfloat16* sh_gu_out;
    // EPI_BF16_COMBINE: the down GEMM of the routed rows (and of the shared expert's T = sh_rows rows, if any) also
    // combines them. cmb_src [rows]: token of each dispatched row (-1: pad); cmb_dest / cmb_gates [T][k]: the rows
    // and gates of each token's choices (-1: dropped); cmb_y [T][h] out; cmb_cnt [T][NT]: arrival counters, zero on
    // entry and zero again when the launch completes.
    const int32_t* cmb_src;
    const int32_t* cmb_dest;
    const float* cmb_gates;
    __nv_bfloat16* cmb_y;
    int* cmb_cnt;
    int cmb_T, cmb_k;
};

// K range of part / expert e in the weight-gradient mapping.
__device__ __forceinline__ void wg_krange(const Params& p, int e, int& k0, int& nkb) {
    if (p.seg) {
        k0 = __ldg(p.seg + e);
        nkb = (__ldg(p.seg + e + 1) - k0) / BK;
    } else {
        k0 = e * p.wg_kchunk;
        nkb = max(0, (min(p.K, k0 + p.wg_kchunk) - k0 + BK - 1) / BK);
    }
}

// sh: the item belongs to the shared expert; K steps kb0 .. kb0 + nkb of BK columns starting at column kx0
struct Work { int e, row0, row1, n, sh, kx0, nkb; };

// Item w of the merged work list: the nr routed items first, then the ns shared-expert items. With the static
// round-robin assignment of items to CTAs, the shorter shared items then fill the routed items' last partial
// wave, and the shared tiles keep their L2 reuse (x rows across n-tiles, a weight tile across m-tiles), which
// spreading them through the list loses. Returns the index within its own list in idx.
__device__ __forceinline__ bool split_item(int w, int nr, int& idx) {
    if (w < nr) { idx = w; return false; }
    idx = w - nr;
    return true;
}

// Work item w -> (expert, rows, n-tile), expert-major, n-tile next, m-tile fastest.
__device__ __forceinline__ Work map_work(const int32_t* sched, int E, int NT, int w) {
    const int32_t* prefix = sched + kSchedHeader;
    int lo = 0, hi = E;                      // find last e with prefix[e] * NT <= w
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)__ldg(prefix + mid) * NT <= w) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int p0 = __ldg(prefix + e), mt = __ldg(prefix + e + 1) - p0;
    const int local = w - p0 * NT;
    const int n = local / mt, m = p0 + local % mt;
    const int4 ent = __ldg(reinterpret_cast<const int4*>(sched + sched_tiles_offset(E)) + m);
    return Work{ent.x, ent.y, ent.z, n, 0, 0, 0};
}

// Merged list of the one-SM kernel: routed items (map_work) and the shared expert's dense 128-row tiles,
// n-tile major, m-tile fastest.
__device__ __forceinline__ Work map_item(const Params& p, int E, int w, int nr, int KB) {
    int idx;
    if (p.wg_E > 0) {                        // weight gradient: expert-major, n-tile next, m-tile fastest
        const int per_e = p.wg_MT * p.NT;
        const int e = w / per_e, rem = w - e * per_e;
        const int n = rem / p.wg_MT, m = rem - n * p.wg_MT;
        int k0, nkb;
        wg_krange(p, e, k0, nkb);
        return Work{e, m * BM, min(m * BM + BM, p.wg_M), n, 0, k0, nkb};
    }
    if (!split_item(w, nr, idx)) {
        Work wk = map_work(p.sched, E, p.NT, idx);
        wk.nkb = KB;
        return wk;
    }
    const int mt = (p.sh_rows + BM - 1) / BM;
    const int n = idx / mt, row0 = (idx % mt) * BM;
    return Work{0, row0, min(row0 + BM, p.sh_rows), n, 1, 0, KB};
}

// bf16 epilogue through TMA stores (EPI_BF16), for a warp whose 32 rows are all valid (row0 .. row0 + 31): 64
// columns at a time in a 4 KB staging box `stg` (1024-byte aligned) in the 128-byte swizzled layout of a
// [32 rows][64 bf16] box (16-byte chunk c of row r at chunk c ^ (r % 8)), stored by one lane at (column, row0) of
// `map`, whose column extent drops the columns past n_valid. Whole lines reach L2 instead of one 16-byte partial
// sector per thread and request. Warps with rows past the tile's valid rows keep the per-thread stores (those
// rows must not be written: they may be the next expert's). The SwiGLU epilogue keeps the per-thread stores:
// its act rows are half as wide, and the staged path measured no faster there.
constexpr int EPI_BF16_BOX_BYTES = 32 * 128;
template <int BN>
__device__ __forceinline__ void store_tile_bf16_tma(const Params& p, const CUtensorMap* map, uint32_t tbase, int n,
                                                    int row0, uint32_t stg) {
    const int lane = threadIdx.x & 31;
    const uint32_t my_row = stg + (uint32_t)lane * 128u;
#pragma unroll 1
    for (int q = 0; q < BN / 64; ++q) {
        float v0[32], v1[32];
        tmem_ld32(tbase + 64 * q, v0);
        tmem_ld32(tbase + 64 * q + 32, v1);
        const int c0 = n * BN + 64 * q;
        if (c0 >= p.n_valid) continue;
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            w[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
            w[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
        }
        if (lane == 0) bulk_wait_read_all();          // the previous box has left the buffer
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 8; ++c)
            st_shared_v4u(my_row + ((uint32_t)(c ^ (lane & 7)) << 4), w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(map, stg, c0, row0);
            bulk_commit();
        }
    }
}

// Epilogue of one accumulator: this thread's TMEM lane (one output row) -> SwiGLU of the packed gate/up
// columns into bf16 act, its backward, or a plain bf16 row, masked to the valid rows and columns.
template <int EPI, int BN>
__device__ __forceinline__ void store_tile(const Params& p, __nv_bfloat16* out, uint32_t tbase, int row, bool live,
                                           int n, __nv_bfloat16* gu = nullptr) {
    if constexpr (EPI == EPI_SWIGLU_BWD) {
        // g, u from the accumulator; da = act gradient (0 past F): s = sigmoid(g),
        // d_g = da u s (1 + g (1 - s)), d_u = da g s, written to columns n*256 + c and n*256 + 128 + c.
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float g[32], u[32];
            tmem_ld32(tbase + 32 * j, g);
            tmem_ld32(tbase + 128 + 32 * j, u);
            const int f0 = n * 128 + 32 * j;
            if (live) {
                __nv_bfloat16* dst = out + (size_t)row * p.ldo + (size_t)n * 256 + 32 * j;
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    Vec16<__nv_bfloat16> da, og, ou;
                    if (f0 + c < p.n_valid) da = ld16(p.d_act + (size_t)row * p.n_valid + f0 + c);
                    else da.v = make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float gv = g[c + i], uv = u[c + i], a = da.get(i);
                        const float sg = 1.f / (1.f + expf(-gv));
                        og.set(i, a * uv * sg * (1.f + gv * (1.f - sg)));
                        ou.set(i, a * gv * sg);
                    }
                    st16(dst + c, og);
                    st16(dst + 128 + c, ou);
                }
            }
        }
    } else if constexpr (EPI == EPI_SWIGLU || EPI == EPI_SWIGLU_SAVE) {
#pragma unroll 1
        for (int j = 0; j < 4; ++j) {
            float g[32], u[32];
            tmem_ld32(tbase + 32 * j, g);
            tmem_ld32(tbase + 128 + 32 * j, u);
            const int f0 = n * 128 + 32 * j;
            if (live) {
                __nv_bfloat16* dst = out + (size_t)row * p.ldo + f0;
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    if (f0 + c < p.n_valid) {
                        Vec16<__nv_bfloat16> o;
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float gv = g[c + i];
                            o.set(i, gv / (1.f + expf(-gv)) * u[c + i]);
                        }
                        st16(dst + c, o);
                    }
                }
                if constexpr (EPI == EPI_SWIGLU_SAVE) {   // pre-activations (f >= F: zero weight rows give zero)
                    __nv_bfloat16* gdst = gu + (size_t)row * (p.NT * 256) + (size_t)n * 256 + 32 * j;
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        Vec16<__nv_bfloat16> og, ou;
#pragma unroll
                        for (int i = 0; i < 8; ++i) { og.set(i, g[c + i]); ou.set(i, u[c + i]); }
                        st16(gdst + c, og);
                        st16(gdst + 128 + c, ou);
                    }
                }
            }
        }
    } else {                                 // EPI_BF16, EPI_BF16_COMBINE
        static_assert(plain_bf16(EPI), "the fp32 epilogue stores through TMA (store_tile_f32_tma)");
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
            float v[32];
            tmem_ld32(tbase + 32 * j, v);
            const int n0 = n * BN + 32 * j;
            if (live) {
                __nv_bfloat16* dst = out + (size_t)row * p.ldo + n0;
#pragma unroll
                for (int c = 0; c < 32; c += 8) {
                    if (n0 + c < p.n_valid) {
                        Vec16<__nv_bfloat16> o;
#pragma unroll
                        for (int i = 0; i < 8; ++i) o.set(i, v[c + i]);
                        st16(dst + c, o);
                    }
                }
            }
        }
    }
}

// fp32 epilogue through TMA stores, one call per epilogue warp (all 32 lanes): the warp's 32 accumulator rows,
// 32 columns at a time, are written into one of its two 4 KB staging boxes at `stg` (1024-byte aligned; the
// warp's n-th box since the kernel began goes to buffer n % 2, `nbox` counting them, so filling one buffer
// overlaps the store of the other and a buffer is refilled only after the store two boxes back has read it)
// in the 128-byte swizzled layout of a [32 rows][32 fp32] box (16-byte chunk c of row r at chunk c ^ (r % 8): the
// eight rows of a store phase hit distinct banks), then one lane stores the box at (column, row0, grp) of `map`,
// whose extents drop the rows and columns past the output. Whole 128-byte lines reach L2, where per-thread row
// stores would send one 16-byte partial sector per request. `live`: the warp holds a valid row (warp-uniform).
constexpr int EPI_BOX_COLS = 32;
constexpr int EPI_STG_BOX_BYTES = 32 * EPI_BOX_COLS * 4;
constexpr int EPI_STG_WARP_BYTES = 2 * EPI_STG_BOX_BYTES;
constexpr int EPI_STG_BYTES = 4 * EPI_STG_WARP_BYTES;
template <int BN>
__device__ __forceinline__ void store_tile_f32_tma(const Params& p, const CUtensorMap* map, uint32_t tbase, int n,
                                                   int row0, int grp, bool zero, bool live, uint32_t stg,
                                                   uint32_t& nbox) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
        float v[32];
        if (zero) {                          // no K steps (an expert without rows): the result is zero
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
        } else {
            tmem_ld32(tbase + 32 * j, v);
        }
        const int n0 = n * BN + 32 * j;
        if (!live || n0 >= p.n_valid) continue;
        if (p.bias) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += n0 + i < p.n_valid ? __ldg(p.bias + n0 + i) : 0.f;
        }
        const uint32_t box = stg + (nbox++ & 1u) * EPI_STG_BOX_BYTES;
        if (lane == 0) bulk_wait_read_but1();          // the box stored from this buffer last time has left it
        __syncwarp();
        const uint32_t my_row = box + (uint32_t)lane * 128u;
#pragma unroll
        for (int c = 0; c < 8; ++c)
            st_shared_v4(my_row + ((uint32_t)(c ^ (lane & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
            tma_store_3d(map, box, n0, row0, grp);
            bulk_commit();
        }
    }
}

// ---------------------------------------------------------------------------------------------------
// Combine fused into the down GEMM's epilogue ("v6 长序列和 MoE", table row "combine": the k expert outputs of a
// token, weighted by their gates, summed back at its position; "专家并行" (formulaic), section "通信与计算的重叠":
// start on the outputs that are ready while the rest is still being computed)
// ---------------------------------------------------------------------------------------------------
// Column block n (256 columns) of y[t] needs block n of each kept expert row of t, and of t's shared-expert row
// when the launch has one: need(t) = kept choices (+ 1). Once an epilogue warp's 32 rows of block n are in memory,
// each row adds one arrival to the counter of (its token, n); the row that brings the count to need(t) makes its
// warp combine that block: y = shared + sum over kept j, ascending, of gate_j * eout[dest_j], fp32 fused
// multiply-adds in that fixed order and one rounding to bf16 -- the arithmetic of moe_combine, so the result is
// bit-identical to it whatever order the tiles finish in. That warp then resets the counter to zero.
// Ordering: a row's values reach memory (the warp's TMA stores completed and proxy-fenced, or the thread's own
// stores), a gpu-scope fence, then the relaxed atomic arrival; the last arriver's warp fences before it reads
// the other rows, through L2 (they were written during this launch).
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

__device__ __forceinline__ int combine_need(const Params& p, int t) {
    int need = p.sh_rows > 0 ? 1 : 0;
    const int32_t* d = p.cmb_dest + (size_t)t * p.cmb_k;
    for (int j = 0; j < p.cmb_k; ++j) need += __ldg(d + j) >= 0 ? 1 : 0;
    return need;
}

// Whole warp: block n of y for up to G tokens tt[g] (< 0: none), one 16-byte chunk of 8 columns per lane, every
// load of the round (shared row and up to KM expert rows per token) in flight before the first use.
template <int G, int KM>
__device__ __forceinline__ void combine_tokens(const Params& p, const int (&tt)[G], int n) {
    const int lane = threadIdx.x & 31, h = p.n_valid, k = p.cmb_k;
    const int c = n * 256 + lane * 8;
    if (c >= h) return;
    int dj[G][KM];
    float gj[G][KM];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            const bool ok = tt[g] >= 0 && j < k;
            dj[g][j] = ok ? __ldg(p.cmb_dest + (size_t)tt[g] * k + j) : -1;
            gj[g][j] = ok ? __ldg(p.cmb_gates + (size_t)tt[g] * k + j) : 0.f;
        }
    uint4 sv[G], v[G][KM];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        sv[g] = make_uint4(0, 0, 0, 0);
        if (tt[g] >= 0 && p.sh_rows > 0) sv[g] = __ldcg(reinterpret_cast<const uint4*>(p.sh_out + (size_t)tt[g] * h + c));
#pragma unroll
        for (int j = 0; j < KM; ++j)
            if (dj[g][j] >= 0) v[g][j] = __ldcg(reinterpret_cast<const uint4*>(p.out + (size_t)dj[g][j] * h + c));
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (tt[g] < 0) continue;
        Vec16<__nv_bfloat16> s;
        s.v = sv[g];
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = p.sh_rows > 0 ? s.get(i) : 0.f;
#pragma unroll
        for (int j = 0; j < KM; ++j) {
            if (dj[g][j] < 0) continue;
            Vec16<__nv_bfloat16> e;
            e.v = v[g][j];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = fmaf(gj[g][j], e.get(i), acc[i]);
        }
        Vec16<__nv_bfloat16> o;
#pragma unroll
        for (int i = 0; i < 8; ++i) o.set(i, acc[i]);
        st16(p.cmb_y + (size_t)tt[g] * h + c, o);
    }
}

// The warp's 32 rows [row0 + lane_base, + 32) of column block n are in memory: one arrival per valid row, then the
// warp combines every block it completed, G tokens per round.
template <int G, int KM>
__device__ __forceinline__ void combine_rounds(const Params& p, unsigned m, int t, int n) {
    const int lane = threadIdx.x & 31;
    while (m) {
        int tt[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            tt[g] = -1;
            if (m) {
                const int src = __ffs(m) - 1;
                m &= m - 1;
                tt[g] = __shfl_sync(0xffffffffu, t, src);
            }
        }
        combine_tokens<G, KM>(p, tt, n);
#pragma unroll
        for (int g = 0; g < G; ++g)
            if (lane == g && tt[g] >= 0) p.cmb_cnt[(size_t)tt[g] * p.NT + n] = 0;
    }
}

__device__ __forceinline__ void combine_arrive(const Params& p, int row0, int row1, bool sh, int n, int lane_base) {
    const int lane = threadIdx.x & 31;
    const int row = row0 + lane_base + lane;
    int t = -1;
    if (row < row1) t = sh ? row : __ldg(p.cmb_src + row);
    bool last = false;
    if (t >= 0) {
        __threadfence();
        const int old = atomicAdd(p.cmb_cnt + (size_t)t * p.NT + n, 1);
        last = old == combine_need(p, t) - 1;
    }
    __threadfence();
    const unsigned m = __ballot_sync(0xffffffffu, last);
    if (!m) return;
    const int k = p.cmb_k;
    if (k <= 2) combine_rounds<4, 2>(p, m, t, n);
    else if (k <= 8) combine_rounds<2, 8>(p, m, t, n);
    else combine_rounds<1, 16>(p, m, t, n);
}

// Tokens with no kept choice and no shared expert receive no arrival: y = 0 for them, written by the epilogue
// warps before their first tile (warp gw of nw).
__device__ __forceinline__ void combine_zero_dropped(const Params& p, int gw, int nw) {
    if (p.sh_rows > 0) return;
    const int lane = threadIdx.x & 31, h = p.n_valid, k = p.cmb_k;
    for (int t = gw; t < p.cmb_T; t += nw) {
        const bool kept = lane < k && __ldg(p.cmb_dest + (size_t)t * k + lane) >= 0;
        if (__any_sync(0xffffffffu, kept)) continue;
        for (int c = lane * 8; c < h; c += 256)
            *reinterpret_cast<uint4*>(p.cmb_y + (size_t)t * h + c) = make_uint4(0, 0, 0, 0);
    }
}

template <int EPI, class CF, bool A8 = false>
__global__ void __launch_bounds__(A8 ? NUM_THREADS_A8 : NUM_THREADS, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2, Params p) {
    constexpr int BN = CF::BN, STAGES = CF::STAGES, B_BYTES = CF::B_BYTES, STAGE_BYTES = CF::STAGE_BYTES;
    constexpr uint32_t kIdesc = idesc_bf16<BN>();
    static_assert((EPI != EPI_SWIGLU && EPI != EPI_SWIGLU_SAVE && EPI != EPI_SWIGLU_BWD) || BN == 256,
                  "the SwiGLU epilogues pair 128 gate with 128 up columns");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase, sB = sbase + STAGES * A_BYTES;
    const uint32_t s8 = sB + STAGES * B_BYTES;                   // A8: e4m3 staging tiles
    const uint32_t s_out = sbase + STAGES * STAGE_BYTES + 1024;   // fp32 epilogue: per-warp store boxes
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES + (A8 ? STAGES * A8_BYTES : 0));
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t mma_done = bar0 + 8u * (2 * STAGES + 4);
    auto raw = [&](int s) { return bar0 + 8u * (2 * STAGES + 5 + s); };   // A8: the TMA copies of a stage landed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 3 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    // with A8 the MMA waits for the converter warps instead of the copies
    auto landed = [&](int s) { return A8 ? raw(s) : full(s); };

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), A8 ? A8_CONVERTER_WARPS : 1);
            mbar_init(empty(s), 1);
            mbar_init(raw(s), 1);
        }
        for (int a = 0; a < 2; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 4); }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.sh_rows) { prefetch_tmap(&tmA2); prefetch_tmap(&tmB2); }
    }
    if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // (launched as a programmatic dependent: everything above overlapped the previous kernel's tail; the tile
    // schedule and the operands are read only from here on)
    pdl_wait();
    pdl_trigger();                           // the next kernel may launch; it waits for this one to complete

    const int E = p.wg_E > 0 ? p.wg_E : __ldg(p.sched + 1);
    const int KB = (p.K + BK - 1) / BK;
    int nr, ns;
    if (p.wg_E > 0) {                                            // weight gradient: every expert's tiles
        nr = p.wg_E * p.wg_MT * p.NT;
        ns = 0;
    } else {
        nr = __ldg(p.sched) * p.NT;                              // routed items
        ns = (p.sh_rows + BM - 1) / BM * p.NT;                   // shared-expert items
    }
    const int total = nr + ns;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0, issued = 0, last_par = 0;
            for (int w = blockIdx.x; w < total && !*abort_flag; w += gridDim.x) {
                const Work wk = map_item(p, E, w, nr, KB);
                const int brow = wk.e * p.b_rows + wk.n * BN;
                const CUtensorMap* ma = wk.sh ? &tmA2 : &tmA;
                const CUtensorMap* mb = wk.sh ? &tmB2 : &tmB;
                bool ok = true;
                for (int kb = 0; kb < wk.nkb; ++kb) {
                    if (!wait_phase(empty(stage), phase ^ 1u, p.wait_limit, abort_flag, p.err, 0x10u)) { ok = false; break; }
                    if constexpr (A8) {
                        mbar_expect_tx(raw(stage), A8_BYTES + B_BYTES);
                        tma_load_2d(s8 + stage * A8_BYTES, ma, wk.kx0 + kb * BK, wk.row0, raw(stage));
                        tma_load_2d(sB + stage * B_BYTES, mb, wk.kx0 + kb * BK, brow, raw(stage));
                    } else {
                        const int kx = wk.kx0 + kb * BK;
                        mbar_expect_tx(full(stage), STAGE_BYTES);
                        tma_load_2d(sA + stage * A_BYTES, ma, p.a_kmod ? kx % p.a_kmod : kx, wk.row0, full(stage));
                        tma_load_2d(sB + stage * B_BYTES, mb, p.b_kmod ? kx % p.b_kmod : kx, brow, full(stage));
                    }
                    issued |= 1u << stage;
                    last_par = (last_par & ~(1u << stage)) | (phase << stage);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            for (int s = 0; s < STAGES; ++s)        // every issued copy has landed before the CTA exits
                if (issued & (1u << s)) drain_phase(landed(s), (last_par >> s) & 1u, p.err, 0x11u);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------------------------ MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            for (int w = blockIdx.x; w < total && !*abort_flag; w += gridDim.x, ++iter) {
                const int a = iter & 1;
                const uint32_t aph = (iter >> 1) & 1;
                if (!wait_phase(tempty(a), aph ^ 1u, p.wait_limit, abort_flag, p.err, 0x20u)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(a * BN);
                const int nkb = map_item(p, E, w, nr, KB).nkb;
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!wait_phase(full(stage), phase, p.wait_limit, abort_flag, p.err, 0x21u)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_s = sA + stage * A_BYTES, b_s = sB + stage * B_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k)
                        umma_bf16(d_tmem, sw128_desc(a_s + k * UK * 2), sw128_desc(b_s + k * UK * 2), kIdesc,
                                  (kb | k) != 0);
                    umma_commit(empty(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit(tfull(a));
            }
            umma_commit(mma_done);                  // all MMAs finished before the columns are freed
            drain_phase(mma_done, 0, p.err, 0x22u);
        }
    } else if (A8 && warp >= 6) {
        // ---------------------------------------------------------------------- e4m3 -> bf16 (warps 6..13)
        // Threads i and i + 128 own row i of the stage, 4 of its 8 16-byte chunks each: codes -> fp32 value * the
        // row's block scale -> bf16, written in the 128-byte-swizzled layout a TMA copy of that bf16 tile would
        // produce (chunk c of row i at chunk c ^ (i % 8)); then a proxy fence so the tensor core sees the generic
        // stores, and one arrival per warp on the stage's full barrier.
        const int i = (threadIdx.x - 192) & (BM - 1), c0 = ((threadIdx.x - 192) >> 7) * 4;
        int stage = 0;
        uint32_t phase = 0;
        for (int w = blockIdx.x; w < total && !*abort_flag; w += gridDim.x) {
            const Work wk = map_item(p, E, w, nr, KB);
            const int row = wk.row0 + i;
            bool ok = true;
            for (int kb = 0; kb < wk.nkb; ++kb) {
                if (!wait_phase(raw(stage), phase, p.wait_limit, abort_flag, p.err, 0x40u)) { ok = false; break; }
                const int col = wk.kx0 + kb * BK;
                const float sc = row < p.a_rows ? __ldg(p.a_scales + (size_t)row * p.a_nblk + (col >> 7)) : 0.f;
                const uint8_t* src = smem + (s8 - sbase) + stage * A8_BYTES + i * BK;
                uint8_t* dst = smem + stage * A_BYTES + i * 128;
#pragma unroll
                for (int c = c0; c < c0 + 4; ++c) {
                    const uint2 q = *reinterpret_cast<const uint2*>(src + 8 * c);
                    const uint32_t qw[2] = {q.x, q.y};
                    uint32_t o[4];
#pragma unroll
                    for (int hw = 0; hw < 4; ++hw) {
                        const __nv_fp8x2_storage_t pr = (__nv_fp8x2_storage_t)((qw[hw >> 1] >> (16 * (hw & 1))) & 0xFFFFu);
                        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
                        const float2 fv = __half22float2(*reinterpret_cast<const __half2*>(&hr));
                        const __nv_bfloat162 bv = __floats2bfloat162_rn(fv.x * sc, fv.y * sc);
                        o[hw] = *reinterpret_cast<const uint32_t*>(&bv);
                    }
                    *reinterpret_cast<uint4*>(dst + ((c ^ (i & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                __syncwarp();
                if (lane == 0) mbar_arrive(full(stage));
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
        }
    } else {
        // ---------------------------------------------------------------------- epilogue (warps 2..5)
        const int lane_base = 32 * (warp & 3);
        int iter = 0;
        uint32_t nbox = 0;                       // fp32 epilogue: store boxes issued by this warp
        if constexpr (EPI == EPI_BF16_COMBINE) combine_zero_dropped(p, blockIdx.x * 4 + (warp & 3), gridDim.x * 4);
        for (int w = blockIdx.x; w < total; w += gridDim.x, ++iter) {
            const int a = iter & 1;
            const uint32_t aph = (iter >> 1) & 1;
            if (!wait_phase(tfull(a), aph, p.wait_limit, abort_flag, p.err, 0x30u)) break;
            tc_fence_after();
            const Work wk = map_item(p, E, w, nr, KB);
            const uint32_t tbase = tmem + (uint32_t)(a * BN) + ((uint32_t)lane_base << 16);
            if constexpr (EPI == EPI_F32) {
                // output box rows: [T] x E logits (group 0), [parts or experts][M] x N, or the de-interleaved
                // gate / up matrices [E][F] x N of the packed gate/up rows
                const CUtensorMap* om = &tmO;
                int orow = wk.row0 + lane_base, grp = 0, lim = wk.row1;
                if (p.wg_E > 0) {
                    grp = wk.e;
                    if (p.wg_gu) {
                        const int b = wk.row0 / BM;
                        om = (b & 1) ? &tmO2 : &tmO;
                        orow = (b >> 1) * BM + lane_base;
                        lim = p.wg_F;
                    }
                }
                store_tile_f32_tma<BN>(p, om, tbase, wk.n, orow, grp, wk.nkb == 0, orow < lim,
                                       s_out + (uint32_t)(warp & 3) * EPI_STG_WARP_BYTES, nbox);
            } else if constexpr (!A8 && plain_bf16(EPI)) {
                const int row0w = wk.row0 + lane_base;
                const bool boxed = row0w + 31 < wk.row1;
                if (boxed) {                             // all 32 rows valid: TMA stores
                    store_tile_bf16_tma<BN>(p, wk.sh ? &tmO2 : &tmO, tbase, wk.n, row0w,
                                            s_out + (uint32_t)(warp & 3) * EPI_BF16_BOX_BYTES);
                } else {
                    const int row = row0w + lane;
                    store_tile<EPI, BN>(p, wk.sh ? p.sh_out : p.out, tbase, row, row < wk.row1, wk.n);
                }
                if constexpr (EPI == EPI_BF16_COMBINE) {
                    // the accumulator is read: hand it back first, then make the rows visible and arrive
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(tempty(a));
                    if (boxed && lane == 0) { bulk_wait_all(); fence_proxy_async_global(); }
                    __syncwarp();
                    combine_arrive(p, wk.row0, wk.row1, wk.sh != 0, wk.n, lane_base);
                    continue;
                }
            } else {
                const int row = wk.row0 + lane_base + lane;
                store_tile<EPI, BN>(p, wk.sh ? p.sh_out : p.out, tbase, row, row < wk.row1, wk.n,
                                    wk.sh ? p.sh_gu_out : p.gu_out);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty(a));
        }
        if (lane == 0) bulk_wait_read_all();           // every box read out of shared memory before the CTA exits
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------------
// 2-SM variant: a cluster of two CTAs computes a 256 x 256 tile with tcgen05.mma.cta_group::2 (M = 256)
// ---------------------------------------------------------------------------------------------------
// The even CTA of the pair (rank 0) issues the MMAs; each CTA holds its own 128 token rows (A) and one half of
// the 256 weight rows (B: rows 0-127 in rank 0, 128-255 in rank 1), so per MMA an SM stages half the weight
// bytes of the one-SM kernel. Every CTA's accumulator holds its 128 rows x all 256 columns, so the epilogue is
// the same. Both CTAs' copies of a stage complete on rank 0's full barrier (TMA .cta_group::2); the MMA commits
// are multicast to both CTAs' barriers; both epilogues arrive on rank 0's accumulator-empty barrier.
// A pair covers two consecutive 128-row tiles of one expert; an odd last tile leaves rank 1 a phantom tile
// whose rows it loads (the partner's, any valid rows) but never stores.
constexpr int PAIR_STAGES = 6;
constexpr int B_HALF_BYTES = 128 * BK * 2;                     // 16 KB
constexpr int PAIR_STAGE_BYTES = A_BYTES + B_HALF_BYTES;       // 32 KB per CTA and stage
constexpr int PAIR_MAX_E = 1024;
constexpr int PAIR_SMEM_BYTES = 1024 + PAIR_STAGES * PAIR_STAGE_BYTES + 256 + (PAIR_MAX_E + 1) * 4;
static_assert(PAIR_SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
// fp32 epilogue (weight-gradient mapping only, which has no pair prefix): the store boxes after the barriers
constexpr int PAIR_STG_OFF = 1024;
constexpr int PAIR_SMEM_BYTES_F32 = 1024 + PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_STG_OFF + EPI_STG_BYTES;
// bf16 epilogues (routed mapping): one store box per epilogue warp after the barriers and the pair prefix
constexpr int PAIR_BOX_OFF = (256 + (PAIR_MAX_E + 1) * 4 + 1023) / 1024 * 1024;
constexpr int PAIR_SMEM_BYTES_BF16 = 1024 + PAIR_STAGES * PAIR_STAGE_BYTES + PAIR_BOX_OFF + 4 * EPI_BF16_BOX_BYTES;
static_assert(PAIR_SMEM_BYTES_BF16 <= 227 * 1024, "shared memory per CTA (bf16 store boxes)");
static_assert(PAIR_SMEM_BYTES_F32 <= 227 * 1024, "shared memory per CTA (fp32 epilogue)");

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Shared-memory address `addr` of this CTA -> the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void st_cluster(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void mbar_complete_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.complete_tx.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait of the pair kernel: a timeout raises the abort flag of both CTAs.
template <bool ACQ_CLUSTER = false>
__device__ __forceinline__ bool wait_phase_pair(uint32_t bar, uint32_t parity, long long limit,
                                                volatile int* abort_flag, uint32_t peer_abort, unsigned* err,
                                                unsigned site) {
    for (long long i = 0; i < limit; ++i) {
        if (ACQ_CLUSTER ? mbar_try_wait_acq_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
    }
    *abort_flag = 1;
    st_cluster(peer_abort, 1u);
    latch_device_error(err, kDevErrTimeout, site);
    return false;
}
// TMA load into this CTA's shared memory whose completion is counted on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int x, int y,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(d_tmem), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on the mbarrier at offset `bar` in both CTAs of the pair once the issued MMAs have completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                 ::"r"(bar), "h"((uint16_t)3)
                 : "memory");
}

// arow: first row this CTA loads; [row0, row1): rows it stores; K steps 0 .. nkb - 1 from column kx0
struct PairWork { int e, arow, row0, row1, n, sh, kx0, nkb; };

// Work item w -> (expert, n-tile, pair of 128-row tiles), expert-major, n-tile next, pair fastest; this CTA
// (rank 0 or 1) takes the first or second tile of the pair. pp: per-expert prefix of pair counts.
__device__ __forceinline__ PairWork map_pair(const int32_t* sched, const int* pp, int E, int NT, int w, int rank) {
    int lo = 0, hi = E;                      // find last e with pp[e] * NT <= w
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if ((long long)pp[mid] * NT <= w) lo = mid; else hi = mid - 1;
    }
    const int e = lo;
    const int np = pp[e + 1] - pp[e];
    const int local = w - pp[e] * NT;
    const int n = local / np, q = local % np;
    const int32_t* prefix = sched + kSchedHeader;
    const int t0 = __ldg(prefix + e), mt = __ldg(prefix + e + 1) - t0;
    const bool has = 2 * q + rank < mt;
    const int4 ent = __ldg(reinterpret_cast<const int4*>(sched + sched_tiles_offset(E)) + t0 + 2 * q + (has ? rank : 0));
    return PairWork{ent.x, ent.y, has ? ent.y : 0, has ? ent.z : 0, n, 0, 0, 0};
}

// Merged list of the 2-SM kernel: routed pair items and the shared expert's dense 256-row pairs (n-tile
// major, pair fastest); a pair whose second tile starts past the shared rows is a phantom for rank 1.
__device__ __forceinline__ PairWork map_pair_item(const Params& p, const int* pp, int E, int w, int nr, int rank,
                                                  int KB) {
    int idx;
    if (p.wg_E > 0) {                        // weight gradient: (expert, n-tile, pair of m-tiles), K = its segment
        const int np = (p.wg_MT + 1) / 2, per_e = np * p.NT;
        const int e = w / per_e, rem = w - e * per_e;
        const int n = rem / np, q = rem - n * np;
        const int m = 2 * q + rank;
        const bool has = m < p.wg_MT;
        int k0, nkb;
        wg_krange(p, e, k0, nkb);
        return PairWork{e, (has ? m : 2 * q) * BM, has ? m * BM : 0, has ? min(m * BM + BM, p.wg_M) : 0, n, 0, k0, nkb};
    }
    if (!split_item(w, nr, idx)) {
        PairWork wk = map_pair(p.sched, pp, E, p.NT, idx, rank);
        wk.nkb = KB;
        return wk;
    }
    const int np = (p.sh_rows + 2 * BM - 1) / (2 * BM);
    const int n = idx / np, q = idx % np;
    const int row0 = 2 * BM * q + BM * rank;
    const bool has = row0 < p.sh_rows;
    return PairWork{0, has ? row0 : 2 * BM * q, has ? row0 : 0, has ? min(row0 + BM, p.sh_rows) : 0, n, 1, 0, KB};
}

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                         const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2, Params p) {
    constexpr int BN = 256, STAGES = PAIR_STAGES;
    constexpr uint32_t kIdesc = idesc_bf16<BN, 2 * BM>();
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sA = sbase, sB = sbase + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * PAIR_STAGE_BYTES);
    const uint32_t bar0 = smem_u32(bars);
    auto full = [&](int s) { return bar0 + 8u * s; };
    auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t mma_done = bar0 + 8u * (2 * STAGES + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* peer_rounds = reinterpret_cast<volatile int*>(tmem_slot + 2);   // rank 1's copy rounds, in rank 0
    int* s_pp = reinterpret_cast<int*>(smem + STAGES * PAIR_STAGE_BYTES + 256);
    const uint32_t s_out = sbase + STAGES * PAIR_STAGE_BYTES + PAIR_STG_OFF;   // fp32 epilogue store boxes
    const uint32_t s_box = sbase + STAGES * PAIR_STAGE_BYTES + PAIR_BOX_OFF;   // bf16 epilogue store boxes

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
        for (int a = 0; a < 2; ++a) { mbar_init(tfull(a), 1); mbar_init(tempty(a), 8); }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        *peer_rounds = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if (p.sh_rows) { prefetch_tmap(&tmA2); prefetch_tmap(&tmB2); }
    }
    // (launched as a programmatic dependent: the barrier set-up above overlapped the previous kernel's tail; the
    // tile schedule and the operands are read only from here on)
    pdl_wait();
    pdl_trigger();                           // the next kernel may launch; it waits for this one to complete
    const int E = p.wg_E > 0 ? p.wg_E : __ldg(p.sched + 1);
    // pair prefix: pp[e + 1] = sum over e' <= e of ceil(tiles_e' / 2) (routed mapping; the fp32 instantiation runs
    // the weight-gradient mapping only, and its store boxes occupy this region)
    if (EPI != EPI_F32 && warp == 2 && p.wg_E == 0) {
        const int32_t* prefix = p.sched + kSchedHeader;
        int carry = 0;
        if (lane == 0) s_pp[0] = 0;
        for (int base = 0; base < E; base += 32) {
            const int e = base + lane;
            int v = e < E ? (__ldg(prefix + e + 1) - __ldg(prefix + e) + 1) >> 1 : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, v, off);
                if (lane >= off) v += t;
            }
            if (e < E) s_pp[e + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
    tc_fence_before();
    cluster_sync_all();                      // barriers initialised and both CTAs' tensor memory allocated
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t peer_abort = map_rank(smem_u32(const_cast<int*>(abort_flag)), rank ^ 1u);

    const int NC = gridDim.x >> 1, cid = blockIdx.x >> 1;
    int nr, ns;
    if (p.wg_E > 0) {                                                   // weight gradient
        nr = p.wg_E * ((p.wg_MT + 1) / 2) * p.NT;
        ns = 0;
    } else {
        nr = s_pp[E] * p.NT;                                            // routed items
        ns = (p.sh_rows + 2 * BM - 1) / (2 * BM) * p.NT;                // shared-expert items
    }
    const int total = nr + ns;
    const int KB = (p.K + BK - 1) / BK;
    int my_rounds = 0;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------------ TMA producer (both CTAs)
            int stage = 0;
            uint32_t phase = 0;
            for (int w = cid; w < total && !*abort_flag; w += NC) {
                const PairWork wk = map_pair_item(p, s_pp, E, w, nr, rank, KB);
                const int brow = wk.e * p.b_rows + wk.n * BN + (int)rank * 128;
                const CUtensorMap* ma = wk.sh ? &tmA2 : &tmA;
                const CUtensorMap* mb = wk.sh ? &tmB2 : &tmB;
                bool ok = true;
                for (int kb = 0; kb < wk.nkb; ++kb) {
                    if (!wait_phase_pair(empty(stage), phase ^ 1u, p.wait_limit, abort_flag, peer_abort, p.err, 0x40u)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_expect_tx(full(stage), 2 * PAIR_STAGE_BYTES);
                    const uint32_t fb = map_rank(full(stage), 0);
                    tma_load_2d_pair(sA + stage * A_BYTES, ma, wk.kx0 + kb * BK, wk.arow, fb);
                    tma_load_2d_pair(sB + stage * B_HALF_BYTES, mb, wk.kx0 + kb * BK, brow, fb);
                    ++my_rounds;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            if (!leader) st_cluster(map_rank(smem_u32(const_cast<int*>(peer_rounds)), 0), (uint32_t)my_rounds);
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------------------------ MMA issuer (rank 0)
            int stage = 0;
            uint32_t phase = 0;
            int iter = 0;
            for (int w = cid; w < total && !*abort_flag; w += NC, ++iter) {
                const int a = iter & 1;
                const uint32_t aph = (iter >> 1) & 1;
                if (!wait_phase_pair<true>(tempty(a), aph ^ 1u, p.wait_limit, abort_flag, peer_abort, p.err, 0x50u))
                    break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(a * BN);
                const int nkb = map_pair_item(p, s_pp, E, w, nr, 0, KB).nkb;
                bool ok = true;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!wait_phase_pair(full(stage), phase, p.wait_limit, abort_flag, peer_abort, p.err, 0x51u)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_s = sA + stage * A_BYTES, b_s = sB + stage * B_HALF_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UK; ++k)
                        umma_bf16_pair(d_tmem, sw128_desc(a_s + k * UK * 2), sw128_desc(b_s + k * UK * 2), kIdesc,
                                       (kb | k) != 0);
                    umma_commit_pair(empty(stage));
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                umma_commit_pair(tfull(a));
            }
            umma_commit_pair(mma_done);             // both CTAs learn when every MMA has finished
        }
    } else {
        // ---------------------------------------------------------------------- epilogue (warps 2..5)
        const int lane_base = 32 * (warp & 3);
        const uint32_t tempty_leader = map_rank(tempty(0), 0);
        int iter = 0;
        uint32_t nbox = 0;                       // fp32 epilogue: store boxes issued by this warp
        if constexpr (EPI == EPI_BF16_COMBINE) combine_zero_dropped(p, blockIdx.x * 4 + (warp & 3), gridDim.x * 4);
        for (int w = cid; w < total; w += NC, ++iter) {
            const int a = iter & 1;
            const uint32_t aph = (iter >> 1) & 1;
            if (!wait_phase_pair(tfull(a), aph, p.wait_limit, abort_flag, peer_abort, p.err, 0x60u)) break;
            tc_fence_after();
            const PairWork wk = map_pair_item(p, s_pp, E, w, nr, rank, KB);
            const uint32_t tbase = tmem + (uint32_t)(a * BN) + ((uint32_t)lane_base << 16);
            if constexpr (EPI == EPI_F32) {
                // as in the one-SM kernel; a phantom tile (row0 == row1) stores nothing
                const CUtensorMap* om = &tmO;
                int orow = wk.row0 + lane_base, grp = 0, lim = wk.row1;
                if (p.wg_E > 0) {
                    grp = wk.e;
                    if (p.wg_gu) {                   // de-interleave: this CTA's m-tile is one packed gate/up block
                        const int b = wk.row0 / BM;
                        om = (b & 1) ? &tmO2 : &tmO;
                        orow = (b >> 1) * BM + lane_base;
                        lim = wk.row0 + lane_base < wk.row1 ? p.wg_F : 0;
                    }
                }
                store_tile_f32_tma<BN>(p, om, tbase, wk.n, orow, grp, wk.nkb == 0, orow < lim,
                                       s_out + (uint32_t)(warp & 3) * EPI_STG_WARP_BYTES, nbox);
            } else if constexpr (plain_bf16(EPI)) {
                const int row0w = wk.row0 + lane_base;
                const bool boxed = row0w + 31 < wk.row1;
                if (boxed) {                             // all 32 rows valid: TMA stores
                    store_tile_bf16_tma<BN>(p, wk.sh ? &tmO2 : &tmO, tbase, wk.n, row0w,
                                            s_box + (uint32_t)(warp & 3) * EPI_BF16_BOX_BYTES);
                } else {
                    const int row = row0w + lane;
                    store_tile<EPI, BN>(p, wk.sh ? p.sh_out : p.out, tbase, row, row < wk.row1, wk.n);
                }
                if constexpr (EPI == EPI_BF16_COMBINE) {
                    // the accumulator is read: hand it back first, then make the rows visible and arrive
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * a);
                    if (boxed && lane == 0) { bulk_wait_all(); fence_proxy_async_global(); }
                    __syncwarp();
                    combine_arrive(p, wk.row0, wk.row1, wk.sh != 0, wk.n, lane_base);
                    continue;
                }
            } else {
                const int row = wk.row0 + lane_base + lane;
                store_tile<EPI, BN>(p, wk.sh ? p.sh_out : p.out, tbase, row, row < wk.row1, wk.n,
                                    wk.sh ? p.sh_gu_out : p.gu_out);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(tempty_leader + 8u * a);
        }
        if (lane == 0) bulk_wait_read_all();           // every box read out of shared memory before the CTA exits
    }
    cluster_sync_all();                      // every role has left its loop; rank 1's round count is in rank 0
    if (warp == 0 && lane == 0 && leader) {
        // Settle the rounds only one CTA issued (possible after an abort), then wait until every copy of both
        // CTAs has landed: rank 1 must not exit while its copies still count on rank 0's barriers.
        const int rl = my_rounds, rp = *peer_rounds;
        for (int n = min(rl, rp); n < max(rl, rp); ++n) {
            if (n < rl) mbar_complete_tx(full(n % STAGES), PAIR_STAGE_BYTES);   // rank 1 never issued round n
            else mbar_expect_tx(full(n % STAGES), PAIR_STAGE_BYTES);            // only rank 1 issued round n
        }
        const int rmax = max(rl, rp);
        for (int s = 0; s < STAGES && s < rmax; ++s) {
            const int last = s + ((rmax - 1 - s) / STAGES) * STAGES;          // last round on stage s
            drain_phase(full(s), (uint32_t)(last / STAGES) & 1u, p.err, 0x41u);
        }
    }
    if (warp == 1 && lane == 0) drain_phase(mma_done, 0, p.err, 0x52u);
    tc_fence_before();
    cluster_sync_all();                      // copies landed, MMAs done, both epilogues finished
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------------------------------
// host: tensor maps and launch
// ---------------------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 tensor [rows, cols] row-major, box [box_rows, 64 columns], 128-byte swizzle, zero fill.
// fp32 output [groups][rows][cols] with row pitch ldo elements, as [32 rows][32 columns] boxes in the 128-byte
// swizzled layout of the epilogue's staging buffers.
static int make_map_out(CUtensorMap* m, float* base, long long groups, long long rows, long long cols, long long ldo) {
    auto fn = encode_fn();
    MOE_REQUIRE(fn, MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    MOE_REQUIRE(base && aligned16(base) && ldo % 4 == 0 && cols <= ldo && groups >= 1 && rows >= 1, MOE_ERR_INVALID_ARG,
                "fp32 output map: base %p ldo %lld cols %lld", (void*)base, ldo, cols);
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)groups};
    cuuint64_t strides[2] = {(cuuint64_t)ldo * 4, (cuuint64_t)rows * ldo * 4};
    cuuint32_t box[3] = {(cuuint32_t)EPI_BOX_COLS, 32, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    MOE_REQUIRE(r == CUDA_SUCCESS, MOE_ERR_CUDA, "cuTensorMapEncodeTiled (fp32 output) failed (%d)", (int)r);
    return MOE_OK;
}

// bf16 output [rows][cols] with row pitch ldo elements, as [32 rows][64 columns] boxes in the 128-byte swizzled
// layout of the epilogue's staging box.
static int make_map_bf16_out(CUtensorMap* m, void* base, long long rows, long long cols, long long ldo) {
    auto fn = encode_fn();
    MOE_REQUIRE(fn, MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    MOE_REQUIRE(base && aligned16(base) && ldo % 8 == 0 && cols <= ldo && rows >= 1, MOE_ERR_INVALID_ARG,
                "bf16 output map: base %p ldo %lld cols %lld rows %lld", base, ldo, cols, rows);
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ldo * 2};
    cuuint32_t box[2] = {64, 32};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    MOE_REQUIRE(r == CUDA_SUCCESS, MOE_ERR_CUDA, "cuTensorMapEncodeTiled (bf16 output) failed (%d)", (int)r);
    return MOE_OK;
}

// Output maps of an fp32 launch: the weight-gradient groups (experts or split-K parts; the gate and up halves
// de-interleaved into two maps) or the dense [a_rows] x n_valid logits; of a plain bf16 launch: the routed
// output [a_rows] and the shared expert's [sh_rows], both n_valid wide with pitch ldo. Other epilogues (and
// absent outputs) take `ma` as a stand-in.
template <int EPI>
static int make_out_maps(const Params& p, long long a_rows, const CUtensorMap& ma, CUtensorMap* o1, CUtensorMap* o2) {
    *o1 = ma;
    *o2 = ma;
    if constexpr (EPI == EPI_F32) {
        if (p.wg_E > 0 && p.wg_gu) {
            if (int rc = make_map_out(o1, p.out_f32, p.wg_E, p.wg_F, p.n_valid, p.ldo)) return rc;
            return make_map_out(o2, p.out2, p.wg_E, p.wg_F, p.n_valid, p.ldo);
        }
        if (p.wg_E > 0) {
            if (int rc = make_map_out(o1, p.out_f32, p.wg_E, p.wg_M, p.n_valid, p.ldo)) return rc;
        } else {
            if (int rc = make_map_out(o1, p.out_f32, 1, a_rows, p.n_valid, p.ldo)) return rc;
        }
        *o2 = *o1;
    }
    if constexpr (plain_bf16(EPI)) {
        if (p.out && a_rows > 0)
            if (int rc = make_map_bf16_out(o1, p.out, a_rows, p.n_valid, p.ldo)) return rc;
        if (p.sh_out && p.sh_rows > 0)
            if (int rc = make_map_bf16_out(o2, p.sh_out, p.sh_rows, p.n_valid, p.ldo)) return rc;
    }
    return MOE_OK;
}

static int make_map(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    auto fn = encode_fn();
    MOE_REQUIRE(fn, MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    MOE_REQUIRE(r == CUDA_SUCCESS, MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) rows=%lld cols=%lld", (int)r,
                rows, cols);
    return MOE_OK;
}

// A second operand set for the same launch: the shared expert's input rows and its packed weights
// (p.sh_rows > 0); otherwise the routed maps are passed twice and never read through the second pair.
struct SharedOperands { const void* a; const void* b; long long b_rows; };

// 2-D uint8 tensor [rows, cols] (e4m3 codes), box [box_rows, 64 columns] = 64 bytes per row, no swizzle.
static int make_map_u8(CUtensorMap* m, const void* base, long long rows, long long cols, int box_rows) {
    auto fn = encode_fn();
    MOE_REQUIRE(fn, MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable from the driver");
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols};
    cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    MOE_REQUIRE(r == CUDA_SUCCESS, MOE_ERR_CUDA, "cuTensorMapEncodeTiled (u8) failed (%d) rows=%lld cols=%lld", (int)r,
                rows, cols);
    return MOE_OK;
}

// The one-SM kernel with an e4m3 A operand dequantised in its prologue (p.a_scales, p.a_nblk, p.a_rows).
template <int EPI>
static int gemm_a8(const void* a8, long long a_rows, const void* b, long long b_rows_total, const Params& p,
                   cudaStream_t s) {
    using CF = Wide;
    static_assert(CF::SMEM_BYTES_A8 <= 227 * 1024, "shared memory per CTA (e4m3 operand)");
    static unsigned long long attr_ctx[64];  // context in which the attribute was set, per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return set_error(MOE_ERR_CUDA, "grouped_gemm (e4m3): no usable current device");
    const unsigned long long ctx = context_id();
    if (ctx == 0 || attr_ctx[dev] != ctx) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, CF, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, CF::SMEM_BYTES_A8);
        if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "grouped_gemm (e4m3) smem attribute: %s", cudaGetErrorString(e));
        attr_ctx[dev] = context_id();
    }
    CUtensorMap ma, mb;
    if (int rc = make_map_u8(&ma, a8, a_rows, p.K, BM)) return rc;
    if (int rc = make_map(&mb, b, b_rows_total, p.K, CF::BN)) return rc;
    static_assert(EPI != EPI_F32, "the e4m3 operand path has no fp32 epilogue");
    grouped_gemm_kernel<EPI, CF, true><<<num_sms(), NUM_THREADS_A8, CF::SMEM_BYTES_A8, s>>>(ma, mb, ma, mb, ma, ma, p);
    return check_launch("grouped_gemm_kernel<up_gate, e4m3 A>");
}

template <int EPI, class CF>
static int gemm(const void* a, long long a_rows, const void* b, long long b_rows_total, const Params& p,
                cudaStream_t s, const SharedOperands& sh = SharedOperands{}) {
    static unsigned long long attr_ctx[64];  // the attribute belongs to the kernel in each device's context
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return set_error(MOE_ERR_CUDA, "grouped_gemm: no usable current device");
    constexpr bool kBox16 = plain_bf16(EPI);
    constexpr int smem_bytes = EPI == EPI_F32 ? 1024 + CF::STAGES * CF::STAGE_BYTES + 1024 + EPI_STG_BYTES
                               : kBox16       ? 1024 + CF::STAGES * CF::STAGE_BYTES + 1024 + 4 * EPI_BF16_BOX_BYTES
                                              : CF::SMEM_BYTES;
    static_assert(smem_bytes <= 227 * 1024, "shared memory per CTA");
    const unsigned long long ctx = context_id();
    if (ctx == 0 || attr_ctx[dev] != ctx) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_kernel<EPI, CF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes);
        if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "grouped_gemm smem attribute: %s", cudaGetErrorString(e));
        attr_ctx[dev] = context_id();
    }
    const long long routed_rows = a_rows;
    if (a_rows == 0) { a = sh.a; a_rows = p.sh_rows; b = sh.b; b_rows_total = sh.b_rows; }   // no routed items
    CUtensorMap ma, mb, ma2, mb2;
    if (int rc = make_map(&ma, a, a_rows, p.a_cols ? p.a_cols : p.K, BM)) return rc;
    if (int rc = make_map(&mb, b, b_rows_total, p.b_cols ? p.b_cols : p.K, CF::BN)) return rc;
    ma2 = ma;
    mb2 = mb;
    if (p.sh_rows > 0) {
        if (int rc = make_map(&ma2, sh.a, p.sh_rows, p.K, BM)) return rc;
        if (int rc = make_map(&mb2, sh.b, sh.b_rows, p.K, CF::BN)) return rc;
    }
    CUtensorMap mo, mo2;
    if (int rc = make_out_maps<EPI>(p, routed_rows, ma, &mo, &mo2)) return rc;
    const cudaError_t le = launch_pdl(grouped_gemm_kernel<EPI, CF>, dim3(num_sms()), dim3(NUM_THREADS), smem_bytes, s, ma,
                                      mb, ma2, mb2, mo, mo2, p);
    if (le != cudaSuccess) return set_error(MOE_ERR_CUDA, "grouped_gemm_kernel launch: %s", cudaGetErrorString(le));
    return check_launch(EPI == EPI_SWIGLU ? "grouped_gemm_kernel<up_gate>"
                        : EPI == EPI_SWIGLU_SAVE ? "grouped_gemm_kernel<up_gate, save>"
                        : EPI == EPI_BF16 ? "grouped_gemm_kernel<bf16>"
                        : EPI == EPI_BF16_COMBINE ? "grouped_gemm_kernel<bf16, combine>"
                        : EPI == EPI_SWIGLU_BWD ? "grouped_gemm_kernel<swiglu_bwd>" : "grouped_gemm_kernel<f32>");
}

// 2-SM kernel: as many pairs as can be resident at once (one CTA per SM), each looping over work items.
template <int EPI>
static int gemm_pair(const void* a, long long a_rows, const void* b, long long b_rows_total, const Params& p,
                     cudaStream_t s, const SharedOperands& sh = SharedOperands{}) {
    static int clusters[64];                 // resident pairs per device, 0 = not yet queried
    static unsigned long long clusters_ctx[64];   // the context they were queried (and the attribute set) in
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return set_error(MOE_ERR_CUDA, "grouped_gemm_pair: no usable current device");
    constexpr bool kBox16 = plain_bf16(EPI);
    constexpr int smem_bytes = EPI == EPI_F32 ? PAIR_SMEM_BYTES_F32 : kBox16 ? PAIR_SMEM_BYTES_BF16 : PAIR_SMEM_BYTES;
    MOE_REQUIRE(EPI != EPI_F32 || p.wg_E > 0, MOE_ERR_INVALID_ARG,
                "grouped_gemm_pair: the fp32 epilogue runs the weight-gradient mapping only");
    const unsigned long long ctx = context_id();
    if (!clusters[dev] || ctx == 0 || clusters_ctx[dev] != ctx) {
        cudaError_t e = cudaFuncSetAttribute(grouped_gemm_pair_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             smem_bytes);
        if (e != cudaSuccess) return set_error(MOE_ERR_CUDA, "grouped_gemm_pair smem attribute: %s", cudaGetErrorString(e));
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (num_sms() / 2));
        cfg.blockDim = dim3(NUM_THREADS);
        cfg.dynamicSmemBytes = smem_bytes;
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<EPI>, &cfg);
        if (e != cudaSuccess || n <= 0)
            return set_error(MOE_ERR_CUDA, "grouped_gemm_pair: no resident cluster of two CTAs (%s)", cudaGetErrorString(e));
        clusters[dev] = std::min(n, num_sms() / 2);
        clusters_ctx[dev] = context_id();
    }
    const long long routed_rows = a_rows;
    if (a_rows == 0) { a = sh.a; a_rows = p.sh_rows; b = sh.b; b_rows_total = sh.b_rows; }   // no routed items
    CUtensorMap ma, mb, ma2, mb2;
    if (int rc = make_map(&ma, a, a_rows, p.K, BM)) return rc;
    if (int rc = make_map(&mb, b, b_rows_total, p.K, 128)) return rc;
    ma2 = ma;
    mb2 = mb;
    if (p.sh_rows > 0) {
        if (int rc = make_map(&ma2, sh.a, p.sh_rows, p.K, BM)) return rc;
        if (int rc = make_map(&mb2, sh.b, sh.b_rows, p.K, 128)) return rc;
    }
    CUtensorMap mo, mo2;
    if (int rc = make_out_maps<EPI>(p, routed_rows, ma, &mo, &mo2)) return rc;
    const cudaError_t le = launch_pdl(grouped_gemm_pair_kernel<EPI>, dim3(2 * clusters[dev]), dim3(NUM_THREADS),
                                      smem_bytes, s, ma, mb, ma2, mb2, mo, mo2, p);
    if (le != cudaSuccess) return set_error(MOE_ERR_CUDA, "grouped_gemm_pair_kernel launch: %s", cudaGetErrorString(le));
    return check_launch(EPI == EPI_SWIGLU ? "grouped_gemm_pair_kernel<up_gate>"
                        : EPI == EPI_SWIGLU_SAVE ? "grouped_gemm_pair_kernel<up_gate, save>"
                        : EPI == EPI_SWIGLU_BWD ? "grouped_gemm_pair_kernel<swiglu_bwd>"
                        : EPI == EPI_F32 ? "grouped_gemm_pair_kernel<f32>"
                        : EPI == EPI_BF16_COMBINE ? "grouped_gemm_pair_kernel<bf16, combine>"
                                                  : "grouped_gemm_pair_kernel<bf16>");
}

// The 2-SM kernel when the average expert has at least four 128-row tiles (an odd tile count costs a
// phantom half tile per expert), otherwise the one-SM kernel.
static bool use_pair(int E, long long rows) { return E <= PAIR_MAX_E && rows >= 4LL * BM * E; }

}  // namespace tc

int ffn_tc_up_gate(const void* buf, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* act,
                   cudaStream_t s, const void* x_sh, int T_sh, const void* packed_sh, void* act_sh, void* gu,
                   void* gu_sh) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    const PackedLayout Ls = packed_layout(1, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    tc::Params p{sched, h, L.Fp / 128, 2 * L.Fp, F, F, static_cast<__nv_bfloat16*>(act), nullptr, nullptr, err,
                 wait_limit(), T_sh, static_cast<__nv_bfloat16*>(act_sh)};
    p.gu_out = static_cast<__nv_bfloat16*>(gu);
    p.sh_gu_out = static_cast<__nv_bfloat16*>(gu_sh);
    const char* b = static_cast<const char*>(packed) + L.up_gate_off;
    const tc::SharedOperands sh{x_sh, packed_sh ? static_cast<const char*>(packed_sh) + Ls.up_gate_off : nullptr,
                                2LL * Ls.Fp};
    if (gu || gu_sh) {
        if (tc::use_pair(E, rows))
            return tc::gemm_pair<tc::EPI_SWIGLU_SAVE>(buf, rows, b, (long long)E * 2 * L.Fp, p, s, sh);
        return tc::gemm<tc::EPI_SWIGLU_SAVE, tc::Wide>(buf, rows, b, (long long)E * 2 * L.Fp, p, s, sh);
    }
    if (tc::use_pair(E, rows)) return tc::gemm_pair<tc::EPI_SWIGLU>(buf, rows, b, (long long)E * 2 * L.Fp, p, s, sh);
    return tc::gemm<tc::EPI_SWIGLU, tc::Wide>(buf, rows, b, (long long)E * 2 * L.Fp, p, s, sh);
}

int ffn_tc_down(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows, void* eout,
                cudaStream_t s, const void* act_sh, int T_sh, const void* packed_sh, void* out_sh) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    const PackedLayout Ls = packed_layout(1, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    using CF = tc::Wide;
    tc::Params p{sched, F, cdiv(h, CF::BN), h, h, h, static_cast<__nv_bfloat16*>(eout), nullptr, nullptr, err,
                 wait_limit(), T_sh, static_cast<__nv_bfloat16*>(out_sh)};
    const char* b = static_cast<const char*>(packed) + L.down_off;
    const tc::SharedOperands sh{act_sh, packed_sh ? static_cast<const char*>(packed_sh) + Ls.down_off : nullptr,
                                (long long)h};
    if (tc::use_pair(E, rows)) return tc::gemm_pair<tc::EPI_BF16>(act, rows, b, (long long)E * h, p, s, sh);
    return tc::gemm<tc::EPI_BF16, CF>(act, rows, b, (long long)E * h, p, s, sh);
}

// The down GEMM with the combine in its epilogue (EPI_BF16_COMBINE): eout and out_sh as ffn_tc_down writes them,
// and y [T][h] = out_sh[t] (if any) + sum over kept j of gates[t][j] eout[dest_row[t][j]]; arrivals [T][cdiv(h, 256)]
// int32 must be zero on entry and are zero again when the launch has completed.
int ffn_tc_down_combine(const void* act, const int32_t* sched, const void* packed, int E, int h, int F, int rows,
                        void* eout, cudaStream_t s, const void* act_sh, int T_sh, const void* packed_sh, void* out_sh,
                        const int32_t* src_token, const int32_t* dest_row, const float* gates, int T, int k, void* y,
                        int32_t* arrivals) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    const PackedLayout Ls = packed_layout(1, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    using CF = tc::Wide;
    tc::Params p{sched, F, cdiv(h, CF::BN), h, h, h, static_cast<__nv_bfloat16*>(eout), nullptr, nullptr, err,
                 wait_limit(), T_sh, static_cast<__nv_bfloat16*>(out_sh)};
    p.cmb_src = src_token;
    p.cmb_dest = dest_row;
    p.cmb_gates = gates;
    p.cmb_y = static_cast<__nv_bfloat16*>(y);
    p.cmb_cnt = arrivals;
    p.cmb_T = T;
    p.cmb_k = k;
    const char* b = static_cast<const char*>(packed) + L.down_off;
    const tc::SharedOperands sh{act_sh, packed_sh ? static_cast<const char*>(packed_sh) + Ls.down_off : nullptr,
                                (long long)h};
    if (tc::use_pair(E, rows)) return tc::gemm_pair<tc::EPI_BF16_COMBINE>(act, rows, b, (long long)E * h, p, s, sh);
    return tc::gemm<tc::EPI_BF16_COMBINE, CF>(act, rows, b, (long long)E * h, p, s, sh);
}

// Up/gate GEMM + SwiGLU on the FP8 send buffer: A = e4m3 codes [rows, h] with per-row, per-128-column fp32
// scales, dequantised to bf16 in the kernel's prologue.
int ffn_tc_up_gate_fp8(const uint8_t* buf8, const float* scales, const int32_t* sched, const void* packed, int E, int h,
                       int F, int rows, void* act, cudaStream_t s) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    tc::Params p{sched, h, L.Fp / 128, 2 * L.Fp, F, F, static_cast<__nv_bfloat16*>(act), nullptr, nullptr, err,
                 wait_limit(), 0, nullptr};
    p.a_scales = scales;
    p.a_nblk = h / 128;
    p.a_rows = rows;
    return tc::gemm_a8<tc::EPI_SWIGLU>(buf8, rows, static_cast<const char*>(packed) + L.up_gate_off,
                                       (long long)E * 2 * L.Fp, p, s);
}

// d_act [rows, F] = d_eout [rows, h] @ W_down[e] per expert, with W_down^T [E][F][h] (backward packing) as
// the K-major operand.
int ffn_tc_down_backward(const void* d_eout, const int32_t* sched, const void* packed_bwd, int E, int h, int F,
                         int rows, void* d_act, cudaStream_t s) {
    const PackedBwdLayout L = packed_bwd_layout(E, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    tc::Params p{sched, h, cdiv(F, 256), F, F, F, static_cast<__nv_bfloat16*>(d_act), nullptr, nullptr, err,
                 wait_limit(), 0, nullptr};
    const char* b = static_cast<const char*>(packed_bwd) + L.down_t_off;
    if (tc::use_pair(E, rows)) return tc::gemm_pair<tc::EPI_BF16>(d_eout, rows, b, (long long)E * F, p, s);
    return tc::gemm<tc::EPI_BF16, tc::Wide>(d_eout, rows, b, (long long)E * F, p, s);
}

// The up/gate GEMM again (g and u are not stored by the forward), its epilogue turning the act gradient into
// the gate and up gradients d_gu [rows, 2 Fp] (packed column order); then d_buf [rows, h] = d_gu @ W_gu[e] with
// W_gu^T [E][h][2Fp] (backward packing) as the K-major operand.
int ffn_tc_up_gate_backward(const void* buf, const void* d_act, const int32_t* sched, const void* packed,
                            const void* packed_bwd, int E, int h, int F, int rows, void* d_gu, void* d_buf,
                            cudaStream_t s) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    const PackedBwdLayout Lb = packed_bwd_layout(E, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    tc::Params p1{sched, h, L.Fp / 128, 2 * L.Fp, F, 2 * L.Fp, static_cast<__nv_bfloat16*>(d_gu), nullptr, nullptr,
                  err, wait_limit(), 0, nullptr, static_cast<const __nv_bfloat16*>(d_act)};
    const char* b1 = static_cast<const char*>(packed) + L.up_gate_off;
    int rc = tc::use_pair(E, rows)
                 ? tc::gemm_pair<tc::EPI_SWIGLU_BWD>(buf, rows, b1, (long long)E * 2 * L.Fp, p1, s)
                 : tc::gemm<tc::EPI_SWIGLU_BWD, tc::Wide>(buf, rows, b1, (long long)E * 2 * L.Fp, p1, s);
    if (rc) return rc;
    return ffn_tc_dbuf(d_gu, sched, packed_bwd, E, h, F, rows, d_buf, s);
}

int ffn_tc_dbuf(const void* d_gu, const int32_t* sched, const void* packed_bwd, int E, int h, int F, int rows,
                void* d_buf, cudaStream_t s) {
    const PackedLayout L = packed_layout(E, h, F, 2);
    const PackedBwdLayout Lb = packed_bwd_layout(E, h, F, 2);
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    tc::Params p2{sched, 2 * L.Fp, cdiv(h, 256), h, h, h, static_cast<__nv_bfloat16*>(d_buf), nullptr, nullptr, err,
                  wait_limit(), 0, nullptr};
    const char* b2 = static_cast<const char*>(packed_bwd) + Lb.gu_t_off;
    if (tc::use_pair(E, rows)) return tc::gemm_pair<tc::EPI_BF16>(d_gu, rows, b2, (long long)E * h, p2, s);
    return tc::gemm<tc::EPI_BF16, tc::Wide>(d_gu, rows, b2, (long long)E * h, p2, s);
}

// Weight gradient of every expert: out[e] [M][N] fp32 = At[:, seg[e] .. seg[e+1]) @ Bt[:, seg[e] .. seg[e+1])^T,
// At [M][ktot] and Bt [N][ktot] bf16 K-major (the experts' rows transposed into 64-aligned column segments).
// gu: At's rows are the packed gate/up order and are written de-interleaved to out (gate) and out2 (up), each
// [E][F][N].
int ffn_tc_weight_grad(const void* At, const void* Bt, long long ktot, const int32_t* seg, int E, int M, int N, int gu,
                       int F, float* out, float* out2, cudaStream_t s) {
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    MOE_REQUIRE(ktot > 0 && ktot % tc::BK == 0 && ktot < (1LL << 31), MOE_ERR_INVALID_ARG,
                "weight gradient: K extent %lld", ktot);
    tc::Params p{seg, (int)ktot, cdiv(N, 256), 0, N, N, nullptr, out, nullptr, err, wait_limit(), 0, nullptr, nullptr,
                 E, cdiv(M, tc::BM), M, seg, gu, F, out2};
    if (cdiv(M, tc::BM) >= 2) return tc::gemm_pair<tc::EPI_F32>(At, M, Bt, N, p, s);   // pairs of m-tiles
    return tc::gemm<tc::EPI_F32, tc::Wide>(At, M, Bt, N, p, s);
}

// Router logits [T, E] fp32 = x [T, h] @ w_rT^T (+ bias), w_rT the K-major [E, h] copy of the router weight,
// `sched` a dense schedule of T rows.
int tc_router_logits(const void* x, const void* w_rT, const float* bias, int T, int h, int E, const int32_t* sched,
                     float* logits, cudaStream_t s) {
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    if (E <= tc::Mid::BN) {
        tc::Params p{sched, h, 1, E, E, E, nullptr, logits, bias, err, wait_limit(), 0, nullptr};
        return tc::gemm<tc::EPI_F32, tc::Mid>(x, T, w_rT, E, p, s);
    }
    tc::Params p{sched, h, cdiv(E, tc::Wide::BN), E, E, E, nullptr, logits, bias, err, wait_limit(), 0, nullptr};
    return tc::gemm<tc::EPI_F32, tc::Wide>(x, T, w_rT, E, p, s);
}

void tc_splitk_plan(int M, int N, int K, int* S, int* kchunk) {
    const long long tiles = (long long)cdiv(M, tc::BM) * cdiv(N, N <= tc::Mid::BN ? tc::Mid::BN : tc::Wide::BN);
    const int S0 = (int)std::min<long long>(std::min(16, cdiv(K, tc::BK)), num_sms() / std::max(1LL, tiles));
    if (S0 < 2) {
        *S = 1;
        *kchunk = cdiv(K, tc::BK) * tc::BK;
        return;
    }
    *kchunk = cdiv(cdiv(K, S0), tc::BK) * tc::BK;
    *S = cdiv(K, *kchunk);
}

int tc_gemm_f32_splitk(const void* a, int M, int a_cols, int a_kmod, const void* b, int N, int b_cols, int b_kmod, int K,
                       int S, int kchunk, float* parts, cudaStream_t s) {
    unsigned* err = device_error_word();
    MOE_REQUIRE(err, MOE_ERR_CUDA, "device error word unavailable");
    MOE_REQUIRE(M > 0 && N > 0 && N % 4 == 0 && K > 0 && S >= 1 && kchunk > 0 && kchunk % tc::BK == 0 &&
                    (long long)(S - 1) * kchunk < K && a_cols % 8 == 0 && b_cols % 8 == 0 && a_kmod % tc::BK == 0 &&
                    b_kmod % tc::BK == 0 && aligned16(a) && aligned16(b) && aligned16(parts),
                MOE_ERR_INVALID_ARG, "tc_gemm_f32_splitk: M=%d N=%d K=%d S=%d kchunk=%d a_cols=%d b_cols=%d", M, N, K, S,
                kchunk, a_cols, b_cols);
    const bool mid = N <= tc::Mid::BN;
    tc::Params p{nullptr, K, mid ? 1 : cdiv(N, tc::Wide::BN), 0, N, N, nullptr, parts, nullptr, err, wait_limit(), 0,
                 nullptr, nullptr, S, cdiv(M, tc::BM), M, nullptr, 0, 0, nullptr};
    p.wg_kchunk = kchunk;
    p.a_cols = a_cols;
    p.b_cols = b_cols;
    p.a_kmod = a_kmod;
    p.b_kmod = b_kmod;
    if (mid) return tc::gemm<tc::EPI_F32, tc::Mid>(a, M, b, N, p, s);
    return tc::gemm<tc::EPI_F32, tc::Wide>(a, M, b, N, p, s);
}

}  // namespace moe
