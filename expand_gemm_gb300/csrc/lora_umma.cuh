// lora_umma.cuh -- inline-PTX wrappers for the Blackwell (sm_100 family)
// asynchronous path: mbarriers, TMA loads (2-D tiles and 1-D bulk
// copies) and tcgen05 (TMEM allocation, UMMA issue/commit, TMEM loads), plus the
// shared-memory and instruction descriptors UMMA takes.
//
// Every wait is bounded: it gives up after `deadline` (a clock64 value) and
// reports failure, so a kernel can raise an error flag and drain instead of
// hanging.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace lora {

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n"
                 :: "r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" :: "r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Waits for the phase with parity `parity` to complete.  Returns false if
// *abort becomes nonzero or the deadline passes (then *abort is set).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, long long deadline)
{
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63) {
            if (*abort) return false;
            if (clock64() > deadline) {
                *abort = 1;
                return false;
            }
        }
    }
}

// mbar_wait_bounded for a thread that runs ahead of its consumers: between
// polls it sleeps `ns` nanoseconds, leaving the issue slots to the warps on
// the critical path.
__device__ __forceinline__ bool mbar_wait_backoff(uint32_t bar, uint32_t parity,
                                                  volatile int *abort, long long deadline,
                                                  uint32_t ns)
{
    while (!mbar_try_wait(bar, parity)) {
        if (*abort) return false;
        if (clock64() > deadline) {
            *abort = 1;
            return false;
        }
        __nanosleep(ns);
    }
    return true;
}

// ---------------------------------------------------------------- CTA pairs
// A cluster of two CTAs on neighbouring SMs driving one tcgen05 MMA with
// M = 256 (cta_group::2): each CTA holds half of A's rows and half of B's
// rows in its own shared memory and its 128 rows of D in its own TMEM.

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

// The shared::cluster address of `smem_addr` (a local shared address) in
// CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive (release, cluster scope) on an mbarrier of another CTA of the
// cluster, given its shared::cluster address.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n"
                 :: "r"(cluster_addr) : "memory");
}

// Every thread of every CTA of the cluster; memory operations before it are
// visible to every thread after it.
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// TMEM allocation shared by the CTA pair: one warp of each CTA executes it.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;\n"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// D[tmem, both CTAs] (+)= A[smem desc, both CTAs] * B[smem desc, both CTAs]^T
// with M = 256: issued by one thread of the even CTA of the pair.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive on the mbarrier at shared::cluster address `bar` (this CTA's or
// its peer's) once every pair UMMA issued so far by this thread has
// completed.
__device__ __forceinline__ void umma_commit_pair(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 :: "r"(bar) : "memory");
}

// ---------------------------------------------------------------- shrink work split

// One of four warp-uniform values, by a warp-uniform index (no local-memory
// array).
__device__ __forceinline__ uint32_t pick4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          int i)
{
    return i == 0 ? a0 : i == 1 ? a1 : i == 2 ? a2 : a3;
}

// The TMA boxes of a tile's x rows.  The tile's nrows (<= 128) sorted tokens
// tk[0 .. nrows) are increasing, so they split into runs of consecutive
// tokens; each run is cut greedily into pieces whose heights are powers of
// two and whose first rows are multiples of their heights (at row j of a run
// ending at e: the largest 2^lg with j a multiple of 2^lg and j + 2^lg <= e).
// Piece word: row | lg << 8 | first token << 11 (tokens below 2^21).  Called
// by a whole warp: the lanes load the tokens (rows lane + 32 i), find the
// run starts by ballots, and walk the runs together; lane 0 writes the
// pieces.  Returns the piece count in every lane.  (Lane 0 alone testing
// each candidate height against the tokens in global memory cost about
// 190 us for a tile of 128 single-token runs: a lora_linear step of the
// large workload's shapes with per-token ids took 1204 us that way, 1017
// this way.)
__device__ __forceinline__ int tile_pieces_warp(const int32_t *tk, int nrows, uint32_t *pieces)
{
    const int lane = threadIdx.x & 31;
    int v[4];
    uint32_t st[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        v[i] = r < nrows ? tk[r] : 0;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = lane + 32 * i;
        int prev = __shfl_up_sync(0xffffffffu, v[i], 1);
        if (i > 0) {
            const int last = __shfl_sync(0xffffffffu, v[i > 0 ? i - 1 : 0], 31);
            if (lane == 0) prev = last;
        }
        st[i] = __ballot_sync(0xffffffffu, r < nrows && (r == 0 || v[i] != prev + 1));
    }
    int n = 0;
    for (int s = 0; s < nrows;) {
        // the run's end: the next run start after s, else nrows
        int e = nrows;
        for (int w = (s + 1) >> 5; w < 4; ++w) {
            uint32_t b = pick4(st[0], st[1], st[2], st[3], w);
            if (w == ((s + 1) >> 5)) b &= ~0u << ((s + 1) & 31);
            if (b != 0u) {
                e = min(nrows, 32 * w + __ffs(int(b)) - 1);
                break;
            }
        }
        const int ts = __shfl_sync(0xffffffffu,
                                   int(pick4(uint32_t(v[0]), uint32_t(v[1]), uint32_t(v[2]),
                                             uint32_t(v[3]), s >> 5)),
                                   s & 31);
        for (int j = s; j < e;) {
            int lg = j == 0 ? 7 : __ffs(j) - 1;
            lg = min(lg, 31 - __clz(e - j));
            if (lane == 0)
                pieces[n] = uint32_t(j) | (uint32_t(lg) << 8) | (uint32_t(ts + (j - s)) << 11);
            ++n;
            j += 1 << lg;
        }
        s = e;
    }
    return n;
}

// Split of the hidden dimension of the tensor-core shrinks: the number of
// chunks (items per tile) that minimises rounds x chunk length (+ a fixed
// cost of about two blocks per item for the pipeline fill and the
// epilogue), with chunks of at least `min_blocks` blocks, for `grid`
// workers.  Every CTA computes the same value.
__device__ __forceinline__ int shrink_kchunks(int tiles, int nk, int grid, int min_blocks)
{
    // 32-bit arithmetic: tiles * 16 and nk are far below 2^31 (T < 2^21).
    int best = 1;
    int best_cost = ((tiles + grid - 1) / grid) * (nk + 2);
    for (int kc = 2; kc <= 16 && nk / kc >= min_blocks; ++kc) {
        const int spc = (nk + kc - 1) / kc;
        const int kce = (nk + spc - 1) / spc;
        const int rounds = (tiles * kce + grid - 1) / grid;
        const int cost = rounds * (spc + 2);
        if (cost < best_cost) {
            best_cost = cost;
            best = kce;
        }
    }
    return best;
}

// ---------------------------------------------------------------- 256-bit store

// One 32-byte global store (the address must be 32-byte aligned).
__device__ __forceinline__ void st_global_v8(void *ptr, const uint32_t (&v)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};\n"
                 :: "l"(ptr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
                    "r"(v[6]), "r"(v[7])
                 : "memory");
}

// As mbar_try_wait / mbar_wait_bounded, with cluster-scope acquire: for
// barriers that threads or tensor cores of another CTA of the cluster
// arrive on.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n.reg .pred p;\n"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_bounded_cluster(uint32_t bar, uint32_t parity,
                                                          volatile int *abort, long long deadline)
{
    for (uint32_t i = 0;; ++i) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((i & 63) == 63) {
            if (*abort) return false;
            if (clock64() > deadline) {
                *abort = 1;
                return false;
            }
        }
    }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];\n"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// 5-D tile load (the row-permuting B map of the tensor-core expand).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, int c3, int c4, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cta.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];\n"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
           "r"(c4), "r"(bar)
        : "memory");
}

// 2-D tile store shared -> global (bulk group; coordinates not negative).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int c0, int c1, uint32_t src)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];\n"
        :: "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(src) : "memory");
}
__device__ __forceinline__ void bulk_commit_group()
{
    asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
}
// Waits until the shared memory read by this thread's bulk stores is free.
__device__ __forceinline__ void bulk_wait_group_read0()
{
    asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed
// (the barrier's count includes this arrival: no pending-count increment).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint32_t bar)
{
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" :: "r"(bar) : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes,
                                             uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Brings the 128-byte line holding p into L2 (no register written, no wait).
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];\n" :: "l"(reinterpret_cast<uint64_t>(p)));
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];\n" :: "l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A's row m in TMEM lane m,
// its K elements packed two per 32-bit column (M = 128).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem,
                                                 uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate)
{
    asm volatile(
        "{\n.reg .pred p;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Arrive on `bar` once every UMMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
                 :: "r"(bar) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of this thread's TMEM lane, without waiting:
// several loads may be in flight before one tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// 16 TMEM lanes x 64 fp32 columns (shape 16x256b, eight repeats along the
// columns), without waiting.  Thread (g, t) = (lane / 4, lane % 4) gets, for
// repeat i, r[4i], r[4i+1] = lane g, columns 8i + 2t and 8i + 2t + 1, and
// r[4i+2], r[4i+3] = lane g + 8, the same columns (the mma.sync
// accumulator layout).
__device__ __forceinline__ void tmem_ld16x256b_x8_nowait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// N consecutive 32-bit columns of this thread's TMEM lane (shape 32x32b).
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N])
{
    static_assert(N == 4 || N == 8 || N == 16 || N == 32, "tmem_st: 4, 8, 16 or 32 columns");
    if constexpr (N == 4) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]) : "memory");
    } else if constexpr (N == 8) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], "
                     "{%1, %2, %3, %4, %5, %6, %7, %8};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),
                        "r"(r[5]), "r"(r[6]), "r"(r[7]) : "memory");
    } else if constexpr (N == 16) {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                     "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),
                        "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]),
                        "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]) : "memory");
    } else {
        asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                     "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
                     "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
                     "%32};\n"
                     :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]),
                        "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]),
                        "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
                        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
                        "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                        "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
    }
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
}

// Shared-memory matrix descriptor: K-major tile of 128-byte rows written
// with the 128-byte swizzle (8-row groups of 1024 bytes, 1024-byte aligned
// tile).  Advancing K by 16 bf16 elements adds 32 bytes to the start.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= uint64_t((saddr & 0x3FFFFu) >> 4);          // start address      [0, 14)
    d |= uint64_t(1) << 16;                           // leading offset     [16, 30) (unused)
    d |= uint64_t(1024 >> 4) << 32;                   // stride offset      [32, 46)
    d |= uint64_t(1) << 46;                           // descriptor version [46, 48)
    d |= uint64_t(2) << 61;                           // 128-byte swizzle   [61, 64)
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n)
{
    return (1u << 4)                         // D format f32      [4, 6)
         | (1u << 7)                         // A format bf16     [7, 10)
         | (1u << 10)                        // B format bf16     [10, 13)
         | (uint32_t(n >> 3) << 17)          // N / 8             [17, 23)
         | (uint32_t(m >> 4) << 24);         // M / 16            [24, 29)
}

// ---------------------------------------------------------------- shrink epilogue

// 16 consecutive fp32 columns of this thread's TMEM lane, without waiting.
__device__ __forceinline__ void tmem_ld16_nowait(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// buf[s][tok, :] += scale * acc for this thread's TMEM lane `tlane` (the
// accumulator of slice s at columns s * RP ...), 64 columns at a time with
// four TMEM loads in flight, added with float4 reductions (red.global.add):
// nothing is read back into the SM, so no load latency is exposed, and an
// element with one owner gets exactly old + scale * acc, as with a plain
// read-modify-write.  tok < 0: nothing is written (the TMEM loads still
// run: they are warp-wide).
__device__ __forceinline__ void shrink_epilogue_row(uint32_t tlane, float *y, int tok, int T,
                                                    int R, int RP, int S, float scale)
{
    const int per_slice = RP / 16;
    const int nch = S * per_slice;
    for (int k0 = 0; k0 < nch; k0 += 4) {
        uint32_t v[4][16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + j;                  // warp-uniform
            if (k < nch)
                tmem_ld16_nowait(tlane + uint32_t((k / per_slice) * RP + (k % per_slice) * 16),
                                 v[j]);
        }
        tmem_wait_ld();
        if (tok < 0) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = k0 + j;
            if (k >= nch) continue;
            const int s = k / per_slice, c = (k % per_slice) * 16;
            float *dst = y + (int64_t(s) * T + tok) * R + c;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (c + 4 * q >= R) continue;
                atomicAdd(reinterpret_cast<float4 *>(dst + 4 * q),
                          make_float4(scale * __uint_as_float(v[j][4 * q]),
                                      scale * __uint_as_float(v[j][4 * q + 1]),
                                      scale * __uint_as_float(v[j][4 * q + 2]),
                                      scale * __uint_as_float(v[j][4 * q + 3])));
            }
        }
    }
}

// Host: encodes a 2-D bf16 tensor map over `rows` rows of `cols` elements
// (row stride in elements) with box {box_cols, box_rows} and the given
// swizzle; false if the driver entry point is missing or rejects it.
bool encode_tile_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                     uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                     CUtensorMapSwizzle swizzle);

// The same over a 2-D fp32 tensor (row stride in elements).
bool encode_tile_map_f32(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols,
                         uint64_t row_stride, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle);

// Host: encodes the B map of the tensor-core expand over a bf16 matrix of
// `rows` rows (a multiple of 64) of `rank` elements, whose boxes of
// `blocks` 64-row blocks land in shared memory with the rows of each block
// permuted: shared row 8i + 2t + e holds global row 16t + 2i + e (i < 8,
// t < 4, e < 2).  Box {box_k, 64 * blocks rows}; false if the driver entry
// point is missing or rejects it.
bool encode_perm_rows_map(CUtensorMap *m, const void *ptr, uint64_t rows, uint32_t rank,
                          uint32_t box_k, uint32_t blocks, CUtensorMapSwizzle swizzle);

}  // namespace lora
