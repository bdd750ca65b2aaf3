// Fused LM-head + Gumbel-max Stage 1 with MXFP4 weights (W4A16) on the tcgen05 tensor cores.
//
// FlashSampling ("Limitations", "Future directions"): low-precision inputs cut the bytes of the
// memory-bound regime.  The weights here are MXFP4 (Open Compute Project Microscaling): E2M1
// elements, two per byte, with one UE8M0 scale per block of 32 elements along K, streamed at
// 0.53 bytes per weight.  The activations stay bf16.  Stage 1 is the same method as the bf16
// kernel (logits on chip, transform, Philox noise, per-tile argmax); only the weight operand
// differs: it is rebuilt as the exact bf16 values E2M1 x 2^(s - 127) in tensor memory, which
// tcgen05.mma kind::f16 reads as its A operand (M = 128 vocabulary rows in the 128 TMEM lanes,
// two bf16 of K per 32-bit column), so the tensor cores run the same bf16 x bf16 -> fp32
// contraction and the rebuilt weights never pass through shared memory.
//
// One thread issues a tcgen05.mma of M = 128, K = 16 about every 105-117 cycles whatever N is
// (measured), while the tensor cores accept several threads' MMAs at once.  A single MMA warp would
// bound the weight stream at decode batch sizes, with every gap between a chunk's MMAs and the next
// (barrier wait, fence, commit) idle.  The CTA therefore runs two independent streams: stream s
// takes the CTA's vocabulary tiles of parity s, with its own MMA warp, converter groups, ring-A
// stages, TMEM slots and accumulators, so the two issue at once.  Each tile is still accumulated
// in a fixed order by one warp.
//
// Warp roles (one persistent CTA per SM):
//   warp 0           bulk-copy producer of the packed weights for both streams: the library's
//                    tiled MXFP4 format (lms_mxfp4_pack) stores each (128-row vocabulary tile,
//                    64-element K chunk) as one contiguous 4352-byte block, 4 KB of codes then 256
//                    bytes of scales, so one cp.async.bulk fills a ring-A stage.
//   warps 1, 2       MMA warps of streams 0 and 1 (warp 1 also allocates TMEM); an elected lane
//                    issues tcgen05.mma (M = 128, N = n_pad batch rows, K = 16 per instruction,
//                    A from TMEM, B = H from shared memory) into the stream's accumulator.
//   warps 3..18      converters, in four groups of four; groups 2s and 2s + 1 serve stream s,
//                    taking its even and odd chunks.  Within a group, warp w (w % 4 = q, the TMEM
//                    lane quarter a warp may access) rebuilds rows 32 q .. 32 q + 31 of each
//                    chunk, one row of 64 weights per lane (byte permutes and one bf16x2 multiply
//                    per pair), and stores them with tcgen05.st into the chunk's TMEM slot.  The
//                    group's first warp also issues the TMA load of the chunk's activations
//                    [n_pad x 64] bf16 into the slot's ring-H stage.  Rebuilding a chunk takes the
//                    SM about 300 cycles of integer-pipe issue once eight or more warps share it,
//                    which bounds this kernel; sixteen warps let each group's barrier waits and
//                    loads overlap the others' rebuilding.
//   warps 19..26     epilogue: as in the bf16 kernel (transform, noise, argmax per tile), over the
//                    tiles in order, each from its stream's accumulator.
// Ring A (packed codes and scales, 4.25 KB a stage, half the stages per stream) is deep so that
// enough weight bytes are in flight to keep HBM busy.  TMEM holds eight rebuilt-weight slots of 32
// columns (four per stream) in columns 0..255 and, from column 256, each stream's accumulators (two
// when 4 n_pad <= 256, so a stream's next tile need not wait for the epilogue; else one); ring H has
// one activation stage per slot, and one tcgen05.commit per chunk frees both.  Every wait is
// bounded in time; a CTA whose wait runs out flags the error, drains its copies and MMAs, poisons
// its remaining candidates (row status 3), frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>

#include "lms.h"
#include "lms_device.cuh"
#include "lms_kernels.h"
#include "tcgen05_common.cuh"

namespace lms {
namespace {

using namespace tc;

constexpr int kMxStreams = 2;
constexpr int kMxGroups = 4;                           // converter groups of four warps, two per stream
constexpr int kMxConvWarps = 4 * kMxGroups;
constexpr int kMxEpiWarps = 8;
constexpr int kMxFirstConv = 3;
constexpr int kMxFirstEpi = kMxFirstConv + kMxConvWarps;
constexpr int kMxThreads = 32 * (kMxFirstEpi + kMxEpiWarps);
// Ring A: stages s * SA/2 .. s * SA/2 + SA/2 - 1 belong to stream s; SA/2 is even, so stage k
// of a stream is only ever read by one of its two groups (the one taking chunks of parity k % 2).
constexpr int kMaxStagesA = 32;
// TMEM: slot t (stream t / 4, the stream's slot t % 4) holds one rebuilt 128 x 64 bf16 chunk in
// columns 32 t .. 32 t + 31; from column 256, each stream's accumulators: two (double-buffered, so a
// stream's next tile need not wait for the epilogue) when 4 n_pad <= 256, else one (n_pad <= 128).
constexpr int kSlotsPerStream = 4;
constexpr int kSlots = kMxStreams * kSlotsPerStream;
constexpr uint32_t kSlotCols = kBK / 2;
constexpr uint32_t kAccCol0 = kSlots * kSlotCols;
constexpr uint32_t kMxTmemCols = 512;
// Longest suspension of a waiting thread per try (it resumes as soon as the phase completes).
constexpr uint32_t kSuspendNs = 100000;
constexpr uint32_t kW4StageBytes = kTileV * kBK / 2;   // 128 rows x 64 codes = 4 KB
constexpr uint32_t kS4StageBytes = 2 * kTileV;         // 2 scale blocks x 128 rows
constexpr uint32_t kAStageBytes = kW4StageBytes + kS4StageBytes;   // one tiled block

struct MxParams {
    SampleArgs a;
    int nk;              // K chunks of 64, ceil(D / 64)
    int n_pad;
    int stages_a;
    int acc_bufs;             // accumulators per stream: 2 when 4 n_pad columns fit beside the slots
    uint32_t h_stage_bytes;   // n_pad * 128
    uint64_t timeout_ns;
    uint32_t debug_flags;
};

// Shared memory (offsets from a 1024-byte aligned base): ring H (activation chunks, one stage per
// TMEM slot, 1024-aligned for the 128-byte swizzle); ring A's packed codes and scales; barriers;
// then the epilogue's buffers.
struct MxLayout {
    uint32_t h_off, a_off, bars_off, misc_off, rows_off, red_off, tr_off, total;
    __host__ __device__ MxLayout(int sa, uint32_t h_stage_bytes, int n_pad) {
        h_off = 0;
        a_off = h_off + kSlots * h_stage_bytes;
        bars_off = a_off + sa * kAStageBytes;
        // fullA, emptyA [SA]; fullC (slot written, count 4), emptyC (slot and its H stage free,
        // one commit), fullH [kSlots]; acc_full[4], acc_empty[4] (stream x buffer), drain[2]
        misc_off = bars_off + (2 * sa + 3 * kSlots + 10) * 8;
        rows_off = (misc_off + 16 + 15) & ~15u;   // misc: tmem slot, error flag
        red_off = rows_off + n_pad * static_cast<uint32_t>(sizeof(RowParams));
        tr_off = red_off + n_pad * 8;
        total = tr_off + kMxEpiWarps * kTrWarpBytes;
    }
};

// E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 as bf16 bit patterns, split into high and low bytes:
// byte m of the 8-byte tables {a, b} is the high (low) byte of magnitude m.
constexpr uint32_t kHiA = 0x3F3F3F00u, kHiB = 0x40404040u;
constexpr uint32_t kLoA = 0xC0800000u, kLoB = 0xC0804000u;

// One 32-bit word of the tiled format (eight elements e0..e7: the magnitude bits of e_k at bits
// 4k..4k+2, the sign of e_k at bit 8k+7 for k < 4 and at bit 8(k-4)+3 for k >= 4) -> eight bf16
// values (pairs in out[0..3], e_2i in the low half of out[i]), times the block scale sc2
// (2^(s - 127) in both halves).  The magnitudes index two 8-entry byte tables (high and low
// bytes of the bf16 value); the sign bits already sit at the top bit of the high byte of their
// element, or four bits below it.
__device__ __forceinline__ void e2m1x8_to_bf16(uint32_t x, __nv_bfloat162 sc2, uint32_t (&out)[4]) {
    const uint32_t mag = x & 0x77777777u;
    uint32_t hb0 = __byte_perm(kHiA, kHiB, mag);
    const uint32_t lb0 = __byte_perm(kLoA, kLoB, mag);
    const uint32_t m1 = mag >> 16;
    uint32_t hb1 = __byte_perm(kHiA, kHiB, m1);
    const uint32_t lb1 = __byte_perm(kLoA, kLoB, m1);
    hb0 |= x & 0x80808080u;                    // signs of e0..e3
    hb1 |= (x << 4) & 0x80808080u;             // signs of e4..e7
    const uint32_t p[4] = {__byte_perm(lb0, hb0, 0x5140), __byte_perm(lb0, hb0, 0x7362),
                           __byte_perm(lb1, hb1, 0x5140), __byte_perm(lb1, hb1, 0x7362)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(&p[i]);
        v = __hmul2(v, sc2);                       // a power of two: exact in the normal range
        out[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

// UE8M0 scale code -> 2^(s - 127) as bf16 in both halves (s = 0: the subnormal 2^-127; s = 255:
// NaN).
__device__ __forceinline__ __nv_bfloat162 ue8m0_to_bf16x2(uint32_t s) {
    const uint32_t h = s == 0 ? 0x0040u : (s == 255 ? 0x7FC0u : (s << 7));
    const uint32_t w = h | (h << 16);
    return *reinterpret_cast<const __nv_bfloat162*>(&w);
}

// Contiguous global -> shared bulk copy completing on an mbarrier (addresses and size 16-byte
// multiples).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// A word of eight E2M1 codes in the logical order (element k in bits 4k..4k+3, sign at bit
// 4k+3) -> the tiled format's word: magnitudes in place, the sign of element k moved to bit
// 8k+7 (k < 4) or 8(k-4)+3 (k >= 4).
__device__ __forceinline__ uint32_t mx_tile_word(uint32_t y) {
    uint32_t out = y & 0x77777777u;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const uint32_t sign = (y >> (4 * k + 3)) & 1u;
        out |= sign << (k < 4 ? 8 * k + 7 : 8 * (k - 4) + 3);
    }
    return out;
}

// The tiled MXFP4 format: block (t, c) at byte (t * nk + c) * kAStageBytes holds the codes of
// rows 128 t .. 128 t + 127 and elements 64 c .. 64 c + 63 (row r at r * 32 as eight
// little-endian words of eight elements each, in mx_tile_word's layout), then the scale codes of
// their two blocks of 32 (block k of row r at 4096 + 128 k + r); rows past V and elements past D
// are zero.  One CTA of 256 threads writes one block.
__global__ void __launch_bounds__(256) mxfp4_pack_kernel(const uint8_t* __restrict__ W4, int64_t ldw4,
                                                          const uint8_t* __restrict__ S, int64_t lds,
                                                          int64_t V, int64_t D, int nk,
                                                          uint8_t* __restrict__ out) {
    const int64_t t = blockIdx.x / nk;
    const int c = static_cast<int>(blockIdx.x - t * nk);
    uint8_t* blk = out + static_cast<int64_t>(blockIdx.x) * kAStageBytes;
    const int i = threadIdx.x;
    {
        const int r = i >> 1, half = i & 1;
        const int64_t v = t * kTileV + r;
        const int64_t byte0 = static_cast<int64_t>(c) * (kBK / 2) + half * 16;   // within the row
        uint8_t piece[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            piece[e] = (v < V && byte0 + e < D / 2) ? W4[v * ldw4 + byte0 + e] : 0;
        uint32_t word[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            word[q] = mx_tile_word(piece[4 * q] | (piece[4 * q + 1] << 8) | (piece[4 * q + 2] << 16) |
                                   (static_cast<uint32_t>(piece[4 * q + 3]) << 24));
        const uint4 w = make_uint4(word[0], word[1], word[2], word[3]);
        *reinterpret_cast<uint4*>(blk + i * 16) = w;
    }
    {
        const int k = i >> 7, r = i & 127;
        const int64_t v = t * kTileV + r;
        const int64_t kb = 2 * static_cast<int64_t>(c) + k;
        blk[kW4StageBytes + i] = (v < V && kb < D / 32) ? S[kb * lds + v] : 0;
    }
}

// 32 TMEM lanes (lane = thread) x 32 consecutive 32-bit columns <- 32 registers per thread, then
// wait until the stores have completed.
__device__ __forceinline__ void tmem_store_32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
        "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// True in exactly one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
    uint32_t pred;
    asm volatile(
        "{\n\t.reg .pred P;\n\t"
        "elect.sync _|P, 0xffffffff;\n\t"
        "selp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(pred));
    return pred != 0;
}

// D[tmem] (+)= A[tmem] * B[smem]^T, bf16 inputs, fp32 accumulate; A is M x 16 in TMEM (row m in
// lane m, two K elements per 32-bit column, the lower K in the low half); issued by one thread.
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

template <bool kWide, bool kPlain>
__global__ void __launch_bounds__(kMxThreads, 1)
    lmhead_mx_kernel(const uint8_t* __restrict__ Wt, const __grid_constant__ CUtensorMap tmH,
                     const MxParams prm) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    const uint32_t base_addr = (raw_addr + 1023u) & ~1023u;
    uint8_t* base = smem_raw + (base_addr - raw_addr);
    const MxLayout L(prm.stages_a, prm.h_stage_bytes, prm.n_pad);

    const SampleArgs& a = prm.a;
    const int SA = prm.stages_a;
    const int n_pad = prm.n_pad;
    const int B = static_cast<int>(a.B);
    const int64_t nt = a.n_tiles;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    const uint32_t bar0 = base_addr + L.bars_off;
    auto fullA = [&](int s) { return bar0 + 8u * s; };
    auto emptyA = [&](int s) { return bar0 + 8u * (SA + s); };
    auto fullC = [&](int t) { return bar0 + 8u * (2 * SA + t); };
    auto emptyC = [&](int t) { return bar0 + 8u * (2 * SA + kSlots + t); };
    auto fullH = [&](int t) { return bar0 + 8u * (2 * SA + 2 * kSlots + t); };
    const uint32_t acc0 = bar0 + 8u * (2 * SA + 3 * kSlots);
    auto accf_bar = [&](int st, int ab) { return acc0 + 8u * (2 * st + ab); };
    auto acce_bar = [&](int st, int ab) { return acc0 + 8u * (4 + 2 * st + ab); };
    auto drain_bar = [&](int st) { return acc0 + 8u * (8 + st); };
    // accumulator (stream st, buffer ab) in TMEM columns kAccCol0 + (st * bufs + ab) * n_pad
    const int bufs = prm.acc_bufs;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + L.misc_off);
    volatile int* err = reinterpret_cast<volatile int*>(base + L.misc_off + 4);
    RowParams* rows = reinterpret_cast<RowParams*>(base + L.rows_off);
    unsigned long long* red = reinterpret_cast<unsigned long long*>(base + L.red_off);

    if (threadIdx.x == 0) {
        for (int k = 0; k < SA; ++k) {
            mbar_init(fullA(k), 1);
            mbar_init(emptyA(k), 4);             // the four warps of the stage's group
        }
        for (int t = 0; t < kSlots; ++t) {
            mbar_init(fullC(t), 4);
            mbar_init(emptyC(t), 1);
            mbar_init(fullH(t), 1);
        }
        for (int st = 0; st < kMxStreams; ++st) {
            for (int ab = 0; ab < 2; ++ab) {
                mbar_init(accf_bar(st, ab), 1);
                mbar_init(acce_bar(st, ab), kMxEpiWarps);
            }
            mbar_init(drain_bar(st), 1);
        }
        *err = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    clear_status_bits(a.status_bits, a.row0);
    if (warp == kMxFirstConv && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmH)) : "memory");
    }
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
        rows[b] = make_row_params(a.temperature, a.seeds, a.positions, a.base_seed, a.offset,
                                  a.row0 + b);
        red[b] = 0ull;
    }
    if (warp == 1) tmem_alloc(base_addr + L.misc_off, kMxTmemCols);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // This CTA's tiles are blockIdx.x + i * gridDim.x, i < my_tiles; stream s takes i = s, s + 2,
    // ...  Chunk u of a stream is K chunk u % nk of its (u / nk)-th tile.  Every role walks its
    // chunks with incremental counters (no division in the loops).
    const int64_t my_tiles = nt > blockIdx.x ? (nt - 1 - blockIdx.x) / gridDim.x + 1 : 0;
    auto tiles_of = [&](int st) { return (my_tiles + 1 - st) / 2; };   // tiles of stream st
    const int half = SA / 2;

    if (warp == 0) {
        // ---------------- bulk-copy producer: packed weights and scales (ring A) ----------------
        // Both streams in lockstep: chunk u of stream 0, then chunk u of stream 1.
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const int64_t n0 = tiles_of(0) * prm.nk, n1 = tiles_of(1) * prm.nk;
            uint32_t issued = 0, issued_parity = 0;
            int stage = 0;                       // stage within each stream's half of ring A
            uint32_t phase = 0;
            int kc = 0;
            int64_t tile0 = blockIdx.x;          // the current tile of stream 0; stream 1's is next
            for (int64_t u = 0; u < n0 && *err == 0; ++u) {
                for (int st = 0; st < kMxStreams; ++st) {
                    if (st == 1 && u >= n1) break;
                    const int k = st * half + stage;
                    if (!mbar_wait_suspend(emptyA(k), phase ^ 1u, prm.timeout_ns, err, kSuspendNs)) {
                        *err = 1;
                        break;
                    }
                    const bool withhold = u == 0 && st == 0 && blockIdx.x == 0 &&
                                          (prm.debug_flags & LMS_DEBUG_WITHHOLD_FIRST_LOAD);
                    if (!withhold) {
                        const int64_t block = (tile0 + st * gridDim.x) * prm.nk + kc;
                        mbar_arrive_expect_tx(fullA(k), kAStageBytes);
                        bulk_load(base_addr + L.a_off + k * kAStageBytes, Wt + block * kAStageBytes,
                                  kAStageBytes, fullA(k), pol_w);
                        issued |= 1u << k;
                        issued_parity = (issued_parity & ~(1u << k)) | (phase << k);
                    }
                }
                if (++stage == half) { stage = 0; phase ^= 1u; }
                if (++kc == prm.nk) { kc = 0; tile0 += 2 * static_cast<int64_t>(gridDim.x); }
            }
            for (int k = 0; k < SA; ++k)
                if (issued & (1u << k))
                    mbar_wait_suspend(fullA(k), (issued_parity >> k) & 1u, prm.timeout_ns, nullptr, kSuspendNs);
        }
    } else if (warp <= kMxStreams) {
        // ---------------- MMA warps: warp 1 + s issues stream s ----------------
        // The whole warp walks the loop, converged, so that the slot counters, TMEM addresses and
        // descriptors stay warp-uniform; one elected lane issues the tcgen05 instructions.
        const int st = warp - 1;
        const bool leader = elect_one();
        const uint32_t idesc = mma_idesc_bf16(n_pad, kTileV);
        bool ok = true;
        int idx = 0;
        uint32_t pt = 0;
        for (int64_t k = 0; k < tiles_of(st) && ok; ++k) {
            const int ab = bufs == 2 ? static_cast<int>(k & 1) : 0;
            const uint32_t round = static_cast<uint32_t>(bufs == 2 ? k >> 1 : k);
            const uint32_t d_tmem = tmem_base + kAccCol0 + static_cast<uint32_t>((st * bufs + ab) * n_pad);
            // the epilogue is done with the tile this accumulator held before
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(acce_bar(st, ab), (round & 1u) ^ 1u,
                                                   prm.timeout_ns, err, kSuspendNs))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            for (int kc = 0; kc < prm.nk; ++kc) {
                const int t = st * kSlotsPerStream + idx;
                // the group announces the slot once its rebuilt weights are stored and the
                // chunk's activations have landed
                if (!__all_sync(0xffffffffu, mbar_wait_suspend(fullC(t), pt, prm.timeout_ns, err, kSuspendNs))) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t a_tmem = tmem_base + static_cast<uint32_t>(t) * kSlotCols;
                const uint64_t bdesc = kmajor_sw128_desc(base_addr + L.h_off + t * prm.h_stage_bytes);
                if (leader) {
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4)
                        mma_bf16_tmem_a(d_tmem, a_tmem + 8u * k4, bdesc + 2u * k4, idesc,
                                        (kc | k4) != 0 ? 1u : 0u);
                    mma_commit(emptyC(t));
                }
                __syncwarp();
                if (++idx == kSlotsPerStream) { idx = 0; pt ^= 1u; }
            }
            if (!ok) break;
            if (leader) mma_commit(accf_bar(st, ab));
            __syncwarp();
        }
        if (!ok && lane == 0) *err = 1;
        if (leader) {
            mma_commit(drain_bar(st));
            mbar_wait_suspend(drain_bar(st), 0, prm.timeout_ns, nullptr, kSuspendNs);
        }
        __syncwarp();
    } else if (warp < kMxFirstEpi) {
        // ---------------- converters ----------------
        // Group G = (warp - 3) / 4 serves stream g = G / 2 and takes its chunks u of parity
        // h = G % 2; the warp's TMEM lane quarter q = warp % 4 gives its rows r = 32 q + lane.  For
        // chunk u (ring-A stage g * SA/2 + u % (SA/2), TMEM slot t = 4 g + u % 4), lane r reads its
        // row's 32 code bytes (64 weights) and two scale codes, rebuilds the 64 bf16 weights as 32
        // bf16x2 words (word c = K elements 2c, 2c + 1) and stores them into TMEM lane r, columns
        // 32 t .. 32 t + 31.
        const int G = (warp - kMxFirstConv) >> 2;
        const int g = G >> 1, h = G & 1;
        const bool h_loader = ((warp - kMxFirstConv) & 3) == 0 && lane == 0;
        const uint64_t pol_h = l2_policy_evict_last();
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(32 * q) << 16);
        const int64_t n_mine = (tiles_of(g) * prm.nk + 1 - h) / 2;
        uint32_t h_issued = 0, h_parity = 0;     // the loader's activation loads, by slot
        // Software pipeline: while chunk u is rebuilt and stored, chunk u + 1's codes are already
        // in registers and its activations on their way.  fetch() takes the next chunk: it waits
        // until that chunk's slot is free, issues its activation load, waits for its ring-A stage
        // and reads the lane's codes and scales.
        // counters of the group's chunks u = h, h + 2, ...: ring-A stage u % (SA/2), slot u % 4 and
        // K chunk u % nk (for the next chunk to fetch and the chunk being stored)
        int stage = h, idx_f = h, idx = h;
        int kc = h < prm.nk ? h : 0;
        uint32_t pa = 0, pt_f = 0, pt = 0;
        uint4 c0 = make_uint4(0, 0, 0, 0), c1 = c0;
        uint32_t s0 = 0, s1 = 0;
        // every wait's outcome is made warp-uniform: tcgen05.st needs the whole warp
        auto fetch = [&]() -> bool {
            const int t = g * kSlotsPerStream + idx_f;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(emptyC(t), pt_f ^ 1u, prm.timeout_ns, err, kSuspendNs)))
                return false;
            if (h_loader) {
                mbar_arrive_expect_tx(fullH(t), prm.h_stage_bytes);
                tma_load_2d(base_addr + L.h_off + t * prm.h_stage_bytes, &tmH, kc * kBK,
                            static_cast<int>(a.row0), fullH(t), pol_h);
                h_issued |= 1u << t;
                h_parity = (h_parity & ~(1u << t)) | (pt_f << t);
            }
            idx_f += 2;
            if (idx_f >= kSlotsPerStream) { idx_f -= kSlotsPerStream; pt_f ^= 1u; }
            kc += 2;
            if (kc >= prm.nk) kc -= prm.nk;
            if (kc >= prm.nk) kc -= prm.nk;
            const int k = g * half + stage;
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(fullA(k), pa, prm.timeout_ns, err, kSuspendNs))) return false;
            const uint8_t* w4 = base + L.a_off + k * kAStageBytes;
            c0 = *reinterpret_cast<const uint4*>(w4 + r * 32);
            c1 = *reinterpret_cast<const uint4*>(w4 + r * 32 + 16);
            s0 = w4[kW4StageBytes + r];
            s1 = w4[kW4StageBytes + kTileV + r];
            // the codes and scales are in registers: this warp is done with the ring-A stage
            __syncwarp();
            if (lane == 0) mbar_arrive(emptyA(k));
            stage += 2;
            if (stage >= half) { stage -= half; pa ^= 1u; }
            return true;
        };
        bool ok = n_mine == 0 || fetch();
        for (int64_t u = 0; u < n_mine && ok; ++u) {
            uint32_t v[32];
            {
                const __nv_bfloat162 sc0 = ue8m0_to_bf16x2(s0), sc1 = ue8m0_to_bf16x2(s1);
                const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
                for (int wd = 0; wd < 8; ++wd) {
                    uint32_t o[4];
                    e2m1x8_to_bf16(cw[wd], wd < 4 ? sc0 : sc1, o);
#pragma unroll
                    for (int i = 0; i < 4; ++i) v[4 * wd + i] = o[i];
                }
            }
            if (u + 1 < n_mine && !fetch()) {
                ok = false;
                break;
            }
            const int t = g * kSlotsPerStream + idx;
            tc_fence_after_sync();
            tmem_store_32(lane_addr + static_cast<uint32_t>(t) * kSlotCols, v);
            // the chunk's activations must have landed too before the slot is announced
            if (!__all_sync(0xffffffffu, mbar_wait_suspend(fullH(t), pt, prm.timeout_ns, err, kSuspendNs))) {
                ok = false;
                break;
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(fullC(t));
            idx += 2;
            if (idx >= kSlotsPerStream) { idx -= kSlotsPerStream; pt ^= 1u; }
        }
        if (!ok && lane == 0) *err = 1;
        // the loader waits (bounded) for its own activation loads still in flight
        if (h_loader)
            for (int t = 0; t < kSlots; ++t)
                if (h_issued & (1u << t))
                    mbar_wait_suspend(fullH(t), (h_parity >> t) & 1u, prm.timeout_ns, nullptr, kSuspendNs);
    } else {
        // ---------------- epilogue ----------------
        const int epi_tid = threadIdx.x - 32 * kMxFirstEpi;
        const int epi_threads = 32 * kMxEpiWarps;
        const int quad = warp & 3;                       // TMEM lanes 32*quad .. 32*quad+31
        const int col_group = (warp - kMxFirstEpi) >> 2;
        float* tr = reinterpret_cast<float*>(base + L.tr_off + (warp - kMxFirstEpi) * kTrWarpBytes);
        int i = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; tile < nt; tile += gridDim.x, ++i) {
            const int st = i & 1;
            const int k = i >> 1;                        // the stream's k-th tile
            const int ab = bufs == 2 ? (k & 1) : 0;
            const uint32_t use_parity = static_cast<uint32_t>(bufs == 2 ? k >> 1 : k) & 1u;
            if (ok) ok = mbar_wait_suspend(accf_bar(st, ab), use_parity, prm.timeout_ns, err, kSuspendNs);
            ok = epi_barrier_and(epi_threads, ok);
            if (!ok) {
                if (epi_tid == 0) *err = 1;
                for (int b = epi_tid; b < B; b += epi_threads) {
                    a.cand_score[b * nt + tile] = -CUDART_INF_F;
                    a.cand_index[b * nt + tile] = kPoisonIndex;
                }
                continue;
            }
            tc_fence_after_sync();
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + kAccCol0 +
                                   static_cast<uint32_t>((st * bufs + ab) * n_pad);
            epilogue_tile_columns<kMxEpiWarps, kWide, kPlain>(a, rows, red, tr, t_row, tile, quad,
                                                              col_group, lane, B);
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(st, ab));
            epi_barrier(epi_threads);
            for (int b = epi_tid; b < B; b += epi_threads) {
                const unsigned long long key = red[b];
                red[b] = 0ull;
                const float sc = unpack_score(key);
                a.cand_score[b * nt + tile] = sc;
                a.cand_index[b * nt + tile] = candidate_index(sc, unpack_index(key));
            }
            epi_barrier(epi_threads);
        }
    }

    pdl_launch_dependents();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, kMxTmemCols);
    }
}

template <bool kWide, bool kPlain>
cudaError_t launch_mx_variant(const uint8_t* Wt, const CUtensorMap& tmH, const MxParams& prm,
                              size_t smem, int grid, cudaStream_t stream) {
    auto kern = lmhead_mx_kernel<kWide, kPlain>;
    const cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kMxThreads, smem, stream>>>(Wt, tmH, prm);
    return cudaGetLastError();
}

}  // namespace

size_t mxfp4_tiled_bytes(int64_t V, int64_t D) {
    return static_cast<size_t>((V + kTileV - 1) / kTileV) * static_cast<size_t>((D + kBK - 1) / kBK) *
           kAStageBytes;
}

cudaError_t launch_mxfp4_pack(const uint8_t* W4, int64_t ldw4, const uint8_t* S, int64_t lds, int64_t V,
                              int64_t D, uint8_t* out, cudaStream_t stream) {
    const int nk = static_cast<int>((D + kBK - 1) / kBK);
    const int64_t blocks = (V + kTileV - 1) / kTileV * nk;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    mxfp4_pack_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(W4, ldw4, S, lds, V, D, nk, out);
    return cudaGetLastError();
}

cudaError_t launch_lmhead_mx(const uint8_t* Wt, const CUtensorMap& tmH, int64_t D, int n_pad, bool wide,
                             uint32_t timeout_ms, uint32_t debug_flags, const SampleArgs& a,
                             cudaStream_t stream) {
    MxParams prm;
    prm.a = a;
    prm.nk = static_cast<int>((D + kBK - 1) / kBK);
    prm.n_pad = n_pad;
    prm.h_stage_bytes = static_cast<uint32_t>(n_pad * kBK * 2);
    if (n_pad > 128) return cudaErrorInvalidValue;       // two accumulators in TMEM columns 256..511
    const uint32_t budget = 227u * 1024u - 1024u;        // opt-in maximum minus alignment slack
    const uint32_t fixed = MxLayout(0, prm.h_stage_bytes, n_pad).total + 2u * kMaxStagesA * 8u;
    // ring A as deep as fits, a multiple of 4 stages from 32 down to 8
    int sa = kMaxStagesA;
    while (fixed + sa * kAStageBytes > budget && sa > 8) sa -= 4;
    if (fixed + sa * kAStageBytes > budget) return cudaErrorInvalidValue;
    prm.stages_a = sa;
    prm.acc_bufs = 4 * n_pad <= static_cast<int>(kMxTmemCols - kAccCol0) ? 2 : 1;
    prm.timeout_ns = static_cast<uint64_t>(timeout_ms) * 1000000ull;
    prm.debug_flags = debug_flags;
    const MxLayout L(sa, prm.h_stage_bytes, n_pad);
    const size_t smem = L.total + 1024;
    const int sms = device_sm_count();
    const int grid = static_cast<int>(a.n_tiles < sms ? a.n_tiles : sms);
    const bool plain = a.bias == nullptr && a.mask == nullptr;
    if (plain)
        return wide ? launch_mx_variant<true, true>(Wt, tmH, prm, smem, grid, stream)
                    : launch_mx_variant<false, true>(Wt, tmH, prm, smem, grid, stream);
    return wide ? launch_mx_variant<true, false>(Wt, tmH, prm, smem, grid, stream)
                : launch_mx_variant<false, false>(Wt, tmH, prm, smem, grid, stream);
}

}  // namespace lms
