// gemv_i8_mma.cu -- small-batch ternary GEMM (M = 2..64 tokens) on the
// fifth-generation tensor cores (integer_engine.md §4.2 with §4.4, batched):
//
//   y[m][r] = sum_g d[r][g] * P[m][r][g],   P[m][r][g] = sum_{i in g} t[r][i] * x[m][i]
//
// Exactness. t is -1/0/+1 and x an int8, both exact fp16 values. The tensor
// core sums one group at a time in fp32 (the group's first K step overwrites
// the accumulator); a group's sum has |P| <= 128 * 128 = 2^14, so every
// partial sum is an integer of magnitude at most 2^14, exact in fp32, and so is
// P + 1.5 * 2^23, which the epilogue forms with one fp32 add: an integer in
// (2^23, 2^24), where consecutive fp32 values are exactly 1 apart, with the bit
// pattern 0x4B400000 + P. The epilogue multiplies that bit pattern by d[r][g] into a wrapping 64-bit
// accumulator per token and at the end subtracts 0x4B400000 * sum_g d[r][g];
// the result is exact modulo 2^64 and therefore exact, since y fits in int64
// (checked on the host).
//
// Mapping. A CTA owns one to four 32-row mask tiles (the MMA's M stays 128;
// the host picks the fewest tiles per CTA that still fill one wave) for all
// groups and all tokens. Warps specialised by role -- 8 producers, two MMA
// warps, a copy warp and 8 folders -- hand work to each other through mbarrier
// rings, with no CTA-wide barrier inside the group loop; work moves between
// them in pairs of groups, so that each wait, fence and arrival serves two
// groups. A warp only touches tensor-memory lanes 32(w%4)..+31, so producers
// and folders are numbered so that w%4 is the row quarter (mask tile) they own.
//   - Producer w (quarter q = w%4, parts 2pp, 2pp+1 with pp = w/4): in its
//     iteration for pair P it expands its 64 weights of each group (group lanes
//     64pp..64pp+63, from the input ring) to fp16, one byte permute per two
//     weights, into A slot P%2 in tensor memory (row = lane, K along the
//     columns), converts two 16-byte activation chunks per group (from the
//     input ring) into B slot P%2 in shared memory, in the canonical K-major
//     layout of 8-row x 16-byte core matrices, and arrives on the input stage's
//     "empty" and the slot's "full" barriers. A producer whose tile the CTA
//     does not own only converts activations.
//   - MMA warp w takes the pairs P = w mod 2, with A/B slot w and D buffer w.
//     When the slot is full and the buffer read back, one thread issues the
//     sixteen K=16 steps of the pair and commits them to the slot's "empty" and
//     the buffer's "full" barriers. An MMA issues every ~50 cycles at N = 64,
//     but any latency in forming its operands sits between one issue and the
//     next, so every operand of a pair is a constant offset from three bases
//     (M = 64: 30.1 -> 28.0 us against a loop that built each descriptor).
//   - Folder f (quarter q = w%4, tokens 32h..32h+31 with h = f/4): for every
//     pair it waits for the D buffer, reads its 32 token columns of each group
//     back from tensor memory, arrives on the buffer's "empty" barrier as soon
//     as the last read has landed, and accumulates them, scaled by d[r][g]
//     (loaded from global memory a pair ahead), into its rows' int64 sums.
//   - A copy warp fills a 3-deep ring of input stages with bulk and tensor
//     (TMA) copies: per pair the mask bytes of the tiles (a tile's two groups
//     are adjacent in the blob) and one 64 x 128 activation box per group
//     (128-byte swizzle, so the producers' 16-byte reads of eight token rows
//     hit eight different bank groups); it refills the stage of pair P with
//     pair P+3 once every producer has arrived on that stage's "empty" barrier.
// Splitting the expansion and the fold over two sets of warps lets each run on
// while the other waits (M = 64 on 13824 x 5120: 33.7 -> 30.2 us; 16 warps that
// both expanded and folded had to pass every hand-off in turn).

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "device_common.cuh"
#include "tg.h"
#include "tg_internal.h"

TGI_DEFINE_DEVICE_ERROR(gemv_mma_take_device_error)

namespace {

using tgi::bulk_copy;
using tgi::mbar_arrive;
using tgi::mbar_expect_tx;
using tgi::mbar_init;
using tgi::smem_u32;

constexpr int kProducerWarps = 8;   // 4 row quarters x 2 parts (64 weights of a group each)
constexpr int kFolderWarps = 8;     // 4 row quarters x 2 token halves (32 tokens each)
constexpr int kMmaWarps = 2;   // MMA issue alternates between two warps (even and odd pairs)
constexpr int kThreads = (kProducerWarps + kMmaWarps + 1 + kFolderWarps) * 32;
constexpr int kFolderWarp0 = kProducerWarps + kMmaWarps + 1;   // producers, MMA warps, copy warp, folders
constexpr int kRowsPerCta = 128;          // the MMA's M: one TMEM lane per row
constexpr int kMaxN = 64;                 // tokens, the MMA's N at most
constexpr int kPair = 2;                  // groups per handshake: work moves between warps in pairs
constexpr int kStages = 3;                // input ring stages (masks and activations of one pair)
constexpr int kSlots = 2;                 // A/B slots, one pair each
constexpr int kDBufs = 2;                 // D buffers, one pair each
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColA = 0;                       // A slots: 128 columns each (2 x 128 fp16 of K per row)
constexpr uint32_t kColD = 128 * kSlots;            // D buffers: 2 x kMaxN columns each
static_assert(kColD + kDBufs * kPair * kMaxN <= kTmemCols, "tensor memory plan");
static_assert(kMaxN == 64, "each folder reads 32 D columns of each group");
static_assert(kSlots == kMmaWarps && kDBufs == kMmaWarps, "MMA warp w owns A/B slot w and D buffer w");
constexpr uint32_t kOffsetBits = 0x4B400000u;   // fp32 bit pattern of 1.5 * 2^23

// Shared-memory plan (dynamic), byte offsets.
constexpr int kKStepBytes = (kMaxN / 8) * 256;         // one K=16 step of B: token octets x 256 B
constexpr int kBBytes = 8 * kKStepBytes;               // one group of B
constexpr int kOffB = 0;                               // kSlots B slots of a pair each
constexpr int kOffStages = kOffB + kSlots * kPair * kBBytes;   // 1024-aligned: the activation box is swizzled
constexpr int kStageMask = 0;                          // masks [tile][group of the pair]: 2 KB per tile
constexpr int kStageX = 8192;                          // activations [group]: 64 tokens x 128 B, 128-byte swizzle
constexpr int kStageXBytes = kMaxN * TG_GROUP;
constexpr int kStageBytes = kStageX + kPair * kStageXBytes;
// mbarriers: input stage full/empty, A/B slot full/empty, D buffer full/empty. Every
// waiter of a barrier is also needed for that barrier's next phase to complete, so no
// waiter can see a phase completed twice over (which would make it wait forever).
constexpr int kBarMFull = 0, kBarMEmpty = kStages, kBarABFull = 2 * kStages, kBarABEmpty = 2 * kStages + kSlots;
constexpr int kBarDFull = 2 * kStages + 2 * kSlots, kBarDEmpty = kBarDFull + kDBufs, kNumBars = kBarDEmpty + kDBufs;
constexpr int kOffAcc = kOffStages + kStages * kStageBytes;   // int64 accumulators [token][row]
constexpr int kOffBar = kOffAcc + kMaxN * kRowsPerCta * 8;
constexpr int kOffSlot = kOffBar + 8 * kNumBars;
constexpr int kSmemBytes = kOffSlot + 16 + 1024;   // + slack to align the base to 1024 bytes
static_assert(kStageBytes % 1024 == 0 && kOffStages % 1024 == 0 && kStageX % 1024 == 0 && kStageXBytes % 1024 == 0,
              "bulk copies need 16-byte and the swizzled activation boxes 1024-byte alignment");

// Shared-memory matrix descriptor, K-major without swizzle: core matrices of
// 8 rows x 16 bytes stored as 128 contiguous bytes, K-adjacent core matrices
// 128 bytes apart (leading byte offset), 8-row groups 256 bytes apart (stride
// byte offset); bit 46 is the descriptor version of this MMA generation.
// The same strides serve every operand tile here.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr)
{
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(128u >> 4) << 16) |
           ((uint64_t)(256u >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor of kind::f16: fp16 A and B, both K-major, fp32 D,
// M = 128, N = n.
__device__ __forceinline__ uint32_t instr_desc(uint32_t n)
{
    return (1u << 4) | ((n >> 3) << 17) | ((uint32_t)(kRowsPerCta >> 4) << 24);
}

__device__ __forceinline__ void mma_a_tmem(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
        ::"r"(d), "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 lanes x 16 columns: thread i writes its v[0..15] into lane (taddr.lane + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15, %16};"
        ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

// 32 lanes x 16 columns: thread i reads lane (taddr.lane + i).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, "
        "%13, %14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]),
          "=r"(v[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Wait for this thread's tensor-memory loads, with the loaded registers passed
// through the wait so that the compiler places no use of them before it (other
// work may sit between the load and the wait).
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]), "+r"(v[7]),
                   "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]), "+r"(v[14]),
                   "+r"(v[15])
                 :
                 : "memory");
}


// 2D tensor (TMA) copy of the box at (x0, y0) of the tensor map into shared
// memory, completing its bytes on the mbarrier.
__device__ __forceinline__ void tensor_copy_2d(uint32_t dst, const CUtensorMap *map, int x0, int y0, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(map), "r"(x0), "r"(y0), "r"(bar)
        : "memory");
}

// Default bound of every wait in this kernel: 2^32 SM clock cycles (about two
// seconds at the part's clocks). The layout's wait_limit overrides it.
constexpr long long kDefaultWaitCycles = 1ll << 32;

// Wait for phase `parity` of an mbarrier: one non-blocking test, then
// suspending waits. Gives up (returns false) after `limit` SM clock cycles, or
// once *abort is set.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort, long long limit)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done)
        return true;
    // each try_wait may suspend the warp until the phase completes, for at most
    // this many nanoseconds (a quarter of the limit's cycles, so that a short
    // limit still runs out on time; at most a millisecond): a waiting warp then
    // issues nothing instead of polling
    const uint32_t hint_ns = (uint32_t)min(limit >> 2, 1000000ll);
    const long long start = clock64();
    while (true) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity), "r"(hint_ns)
            : "memory");
        if (done)
            return true;
        if (*abort || clock64() - start > limit)
            return false;
    }
}

// Wait, before the CTA frees its tensor memory and exits, for an asynchronous
// operation this CTA started (bulk and tensor copies into its shared memory,
// MMAs committed to an mbarrier) to signal phase `parity` of `bar`. Such an
// operation always ends, so this wait ignores the abort flag and the caller's
// limit; it is still bounded (the default limit) and sets the error word if it
// runs out.
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity)
{
    const long long start = clock64();
    while (!tgi::mbar_test(bar, parity)) {
        if (clock64() - start > kDefaultWaitCycles) {
            atomicExch(&tgi_device_error_word, 1);
            return;
        }
    }
}

// fp16 (+1, -1, 0) of weight codes f = W_nonzero | W_negative << 1 held in
// nibbles 1 and 3 of the selector: byte 0 of the table is 0x00 (the low byte
// of every value, and the high byte for f = 0), byte 1 is 0x3C (+1: 0x3C00),
// byte 3 is 0xBC (-1: 0xBC00).
__device__ __forceinline__ uint32_t fp16_pair(uint32_t sel) { return __byte_perm(0xBC003C00u, 0u, sel); }

// Eight int8 activations -> eight exact fp16 values: the bytes x ^ 0x80 =
// x + 128 sit under the exponent byte 0x64 (fp16 0x64bb is 1024 + bb exactly),
// then 1152 is subtracted (exact: the result is the integer x).
__device__ __forceinline__ uint32_t fp16x2_sub1152(uint32_t v)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(0x64806480u));
    return r;
}

__device__ __forceinline__ uint4 fp16_of_int8x8(uint2 v)
{
    const uint32_t lo = v.x ^ 0x80808080u, hi = v.y ^ 0x80808080u;
    return make_uint4(fp16x2_sub1152(__byte_perm(lo, 0x64646464u, 0x5140)),
                      fp16x2_sub1152(__byte_perm(lo, 0x64646464u, 0x7362)),
                      fp16x2_sub1152(__byte_perm(hi, 0x64646464u, 0x5140)),
                      fp16x2_sub1152(__byte_perm(hi, 0x64646464u, 0x7362)));
}

// acc + (int64)a * b, wrapping modulo 2^64.
__device__ __forceinline__ uint64_t mad_wide(uint32_t a, int32_t b, uint64_t acc)
{
    uint64_t r;
    asm("mad.wide.s32 %0, %1, %2, %3;" : "=l"(r) : "r"(a), "r"(b), "l"(acc));
    return r;
}

// Expand one mask word (16 weights, lanes 16u + 4j + b in bits 8b + 2j, 8b + 2j + 1)
// into 8 fp16 pairs: out[2j] holds lanes 4j, 4j + 1 and out[2j + 1] lanes 4j + 2, 4j + 3.
__device__ __forceinline__ void expand_word(uint32_t w, uint32_t *out)
{
#pragma unroll
    for (int j = 0; j < 4; j++) {
        const uint32_t m = w & (0x03030303u << (2 * j));
        const uint32_t s01 = j < 2 ? m << (4 - 2 * j) : m >> (2 * j - 4);   // codes of bytes 0, 1 -> nibbles 1, 3
        out[2 * j] = fp16_pair(s01);
        out[2 * j + 1] = fp16_pair(m >> (12 + 2 * j));                    // bytes 2, 3 -> nibbles 1, 3
    }
}

// Q1_0: expand one word of sign bits (lane 4j + b in bit 8b + j, set for +1)
// into 8 fp16 pairs, out[2j] = lanes 4j, 4j + 1 and out[2j + 1] = lanes
// 4j + 2, 4j + 3. Selector nibbles 1 and 3 are 1 + 2 * bit: table byte 1 is
// 0xBC (-1: 0xBC00), byte 3 is 0x3C (+1: 0x3C00), byte 0 the zero low byte.
__device__ __forceinline__ void expand_word_q1(uint32_t w, uint32_t *out)
{
#pragma unroll
    for (int j = 0; j < 8; j++) {
        const uint32_t s01 = ((j <= 5 ? w << (5 - j) : w >> (j - 5)) & 0x2020u) | 0x1010u;   // bits j, 8 + j
        const uint32_t s23 = ((w >> (11 + j)) & 0x2020u) | 0x1010u;                          // bits 16 + j, 24 + j
        out[2 * j] = __byte_perm(0x3C00BC00u, 0u, s01);
        out[2 * j + 1] = __byte_perm(0x3C00BC00u, 0u, s23);
    }
}

// Folds of a group's accumulator bits (0x4B400000 + P) into the outputs:
// kFoldNarrow: frac = 0 and every |d| <= kNarrowMaxScale, so kBlock groups of
//   exact P * d sum below 2^31 in magnitude: one wrapping 32-bit multiply-add
//   per value and a 64-bit flush every kBlock groups;
// kFoldWide: frac = 0, larger scales: one 64-bit multiply-add per value and
//   0x4B400000 * sum_g d subtracted at the end;
// kFoldFloor: frac > 0: each group's P * d is floored by 2^frac on its own
//   (integer_engine.md §4.1/§4.2 arshift) before it is added.
constexpr int kFoldNarrow = 0, kFoldWide = 1, kFoldFloor = 2;
constexpr int kBlock = 4;
constexpr int64_t kNarrowMaxScale = 32767;   // 4 * 2^14 * 32767 < 2^31
static_assert((int64_t)kBlock * 16384 * kNarrowMaxScale < ((int64_t)1 << 31), "narrow fold bound");

template <bool kQ1, int kFold>
__global__ void __launch_bounds__(kThreads, 1)
gemv_i8_mma_kernel(const unsigned char *__restrict__ masks, const unsigned char *__restrict__ scales,
                   const __grid_constant__ CUtensorMap xmap, int64_t *__restrict__ y, int N, int G, int tiles,
                   int M, int frac, int ctiles, long long wait_limit)
{
    constexpr bool kNarrow = kFold == kFoldNarrow;
    constexpr uint32_t kMaskBytes = kQ1 ? 512u : 1024u;   // mask bytes of one (tile, group)
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ volatile int abort_flag;   // set when a bounded wait gave up
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const uint32_t nmma = (uint32_t)((M + 15) & ~15);
    const int tiles_here = min(ctiles, tiles - (int)blockIdx.x * ctiles);

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kOffBar;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    auto *slot = reinterpret_cast<volatile uint32_t *>(smem + kOffSlot);

    // --- set-up: zero the B slots (tokens M.. stay zero) and the accumulators, barriers, TMEM
    for (int i = tid; i < kOffStages / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem)[i] = make_uint4(0, 0, 0, 0);
    for (int i = tid; i < kMaxN * kRowsPerCta * 8 / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + kOffAcc)[i] = make_uint4(0, 0, 0, 0);
    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < kStages; i++) {
            mbar_init(bar(kBarMFull + i), 1);
            mbar_init(bar(kBarMEmpty + i), kProducerWarps);
        }
        for (int i = 0; i < kSlots; i++) {
            mbar_init(bar(kBarABFull + i), kProducerWarps);
            mbar_init(bar(kBarABEmpty + i), 1);
        }
        for (int i = 0; i < kDBufs; i++) {
            mbar_init(bar(kBarDFull + i), 1);
            mbar_init(bar(kBarDEmpty + i), kFolderWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(sbase + kOffSlot),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = *slot;

    // A bounded wait; once any thread has given up, the others stop waiting too.
    auto wait = [&](int i, uint32_t parity) {
        if (!mbar_wait(bar(i), parity, &abort_flag, wait_limit) && !abort_flag) {
            atomicExch(&tgi_device_error_word, 1);
            abort_flag = 1;
        }
    };

    const int npairs = (G + kPair - 1) / kPair;
    if (warp == kProducerWarps + kMmaWarps) {
        // ---------------- copy warp: inputs of pair P -> stage P % kStages ----------------
        auto copy_inputs = [&](int P) {
            const int st = P % kStages, g0 = kPair * P;
            const int ng = min(kPair, G - g0);
            const uint32_t sdst = sbase + kOffStages + st * kStageBytes;
            const uint32_t b = bar(kBarMFull + st);
            if (lane == 0)
                mbar_expect_tx(b, (uint32_t)(tiles_here * ng) * kMaskBytes + (uint32_t)(ng * kStageXBytes));
            __syncwarp();
            if (lane < tiles_here) {
                // the pair's groups of one tile are adjacent in the blob
                const size_t unit = (size_t)(blockIdx.x * ctiles + lane) * G + g0;
                bulk_copy(sdst + kStageMask + lane * 2048, masks + unit * kMaskBytes, (uint32_t)ng * kMaskBytes, b);
            } else if (lane >= 32 - ng) {
                // 64 token rows x 128 bytes of group g0 + h (rows from M on read as zero)
                const int h = 31 - lane;
                tensor_copy_2d(sdst + kStageX + h * kStageXBytes, &xmap, (g0 + h) * TG_GROUP, 0, b);
            }
            __syncwarp();
        };
        int issued = 0;   // pairs whose copies are in flight or landed: 0 .. issued - 1
        for (int P = 0; P < min(npairs, kStages); P++, issued++)
            copy_inputs(P);
        for (int P = 0; P + kStages < npairs; P++) {
            // every producer has read stage P % kStages
            if (lane == 0)
                wait(kBarMEmpty + P % kStages, (uint32_t)(P / kStages) & 1u);
            __syncwarp();
            if (__shfl_sync(0xffffffffu, abort_flag, 0))
                break;
            copy_inputs(P + kStages);
            issued++;
        }
        // every copy this warp started has landed before the CTA exits (after a
        // give-up, some stages were never read): the last filling of each stage
        if (lane == 0)
            for (int P = max(issued - kStages, 0); P < issued; P++)
                mbar_drain(bar(kBarMFull + P % kStages), (uint32_t)(P / kStages) & 1u);
        __syncwarp();
    } else if (warp >= kProducerWarps && warp < kProducerWarps + kMmaWarps) {
        // ---------------- MMA warp w: pairs P = w mod 2, A/B slot and D buffer w ----------------
        const uint32_t idesc = instr_desc(nmma);
        const int w = warp - kProducerWarps;
        if (lane == 0) {
            int last = -1;   // the last pair whose MMAs this warp committed
            for (int P = w; P < npairs && !abort_flag; P += kMmaWarps) {
                const uint32_t par = (uint32_t)(P / kMmaWarps) & 1u;
                wait(kBarABFull + w, par);
                wait(kBarDEmpty + w, par);   // read back by every folder
                if (abort_flag)
                    break;
                fence_after_sync();
                const int ng = min(kPair, G - kPair * P);
                // every operand address of the pair is a constant offset from these three, so no
                // latency sits between one MMA's issue and the next
                const uint32_t d0 = tmem + kColD + (uint32_t)(kPair * kMaxN * w);
                const uint32_t a0 = tmem + kColA + (uint32_t)(128 * w);
                const uint64_t b0 = smem_desc(sbase + kOffB + (uint32_t)(kPair * w * kBBytes));
#pragma unroll
                for (int h = 0; h < kPair; h++) {
                    if (h < ng) {
#pragma unroll
                        for (int ks = 0; ks < 8; ks++)
                            mma_a_tmem(d0 + (uint32_t)(kMaxN * h), a0 + (uint32_t)(64 * h + 8 * ks),
                                       b0 + (uint64_t)((h * kBBytes + ks * kKStepBytes) >> 4), idesc, ks > 0 ? 1u : 0u);
                    }
                }
                mma_commit(bar(kBarABEmpty + w));
                mma_commit(bar(kBarDFull + w));
                last = P;
            }
            // the MMAs this warp issued have completed before tensor memory is freed
            // (after a give-up their D buffer may never have been read)
            if (last >= 0)
                mbar_drain(bar(kBarDFull + w), (uint32_t)(last / kMmaWarps) & 1u);
        }
        __syncwarp();
    } else if (warp < kProducerWarps) {
        // ---------------- producer warps: A (expanded weights) and B (converted activations) ----------------
        const int q = warp & 3, pp = warp >> 2;   // row quarter; parts 2 pp, 2 pp + 1 (64 weights of a group)
        const bool rows_q = q < ctiles;
        const int tile = blockIdx.x * ctiles + q;
        const bool tile_ok = rows_q && tile < tiles;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        // activation chunks: token xn, 16-byte chunks j16 and j16 + 4 of each group, from the
        // stage's swizzled box (chunk j of row n sits at chunk j ^ (n & 7))
        const int xn = (warp & 7) * 8 + (lane & 7);
        const bool x_ok = xn < M;
        const int j16 = lane >> 3;
        const int xoff0 = kStageX + xn * TG_GROUP + ((j16 ^ (xn & 7)) << 4);
        const int xoff1 = kStageX + xn * TG_GROUP + (((j16 + 4) ^ (xn & 7)) << 4);
        // this thread's 64 weights of a group: 16 bytes (Q1: 8) of its row in the stage
        const unsigned char *mrow = kQ1 ? smem + kOffStages + kStageMask + q * 2048 + lane * 16 + 8 * pp
                                        : smem + kOffStages + kStageMask + q * 2048 + pp * 512 + lane * 16;
        const uint32_t abase = tmem + lane_off + kColA + 32u * (uint32_t)pp;
        unsigned char *bdst0 = smem + kOffB + j16 * kKStepBytes + (xn >> 3) * 256 + (xn & 7) * 16;
        unsigned char *bdst1 = bdst0 + 4 * kKStepBytes;

        int st = 0;
        uint32_t st_par = 0;
#pragma unroll 1
        for (int P = 0; P < npairs; P++) {
            const int sl = P & 1;
            const uint32_t sl_par = (uint32_t)(P >> 1) & 1u;
            const int ng = min(kPair, G - kPair * P);
            if (P >= kSlots)   // A/B slot free: the MMAs of pair P - 2 are done
                wait(kBarABEmpty + sl, sl_par ^ 1u);
            wait(kBarMFull + st, st_par);
#pragma unroll
            for (int h = 0; h < kPair; h++) {
                if (h < ng) {
                    if (rows_q) {
                        uint4 mw = make_uint4(0, 0, 0, 0);
                        if (tile_ok) {
                            const unsigned char *mp = mrow + (size_t)st * kStageBytes + h * kMaskBytes;
                            if (kQ1) {
                                const uint2 m2 = *reinterpret_cast<const uint2 *>(mp);
                                mw = make_uint4(m2.x, m2.y, 0u, 0u);
                            } else {
                                mw = *reinterpret_cast<const uint4 *>(mp);
                            }
                        }
                        const uint32_t at = abase + 128u * (uint32_t)sl + 64u * (uint32_t)h;
                        uint32_t a[16];
                        if (kQ1) {
                            expand_word_q1(mw.x, a);
                            tmem_st16(at, a);
                            expand_word_q1(mw.y, a);
                            tmem_st16(at + 16u, a);
                        } else {
                            expand_word(mw.x, a);
                            expand_word(mw.y, a + 8);
                            tmem_st16(at, a);
                            expand_word(mw.z, a);
                            expand_word(mw.w, a + 8);
                            tmem_st16(at + 16u, a);
                        }
                    }
                    if (x_ok) {
                        const unsigned char *xs = smem + kOffStages + (size_t)st * kStageBytes + h * kStageXBytes;
                        const uint4 xv0 = *reinterpret_cast<const uint4 *>(xs + xoff0);
                        const uint4 xv1 = *reinterpret_cast<const uint4 *>(xs + xoff1);
                        const int bo = (sl * kPair + h) * kBBytes;
                        *reinterpret_cast<uint4 *>(bdst0 + bo) = fp16_of_int8x8(make_uint2(xv0.x, xv0.y));
                        *reinterpret_cast<uint4 *>(bdst0 + bo + 128) = fp16_of_int8x8(make_uint2(xv0.z, xv0.w));
                        *reinterpret_cast<uint4 *>(bdst1 + bo) = fp16_of_int8x8(make_uint2(xv1.x, xv1.y));
                        *reinterpret_cast<uint4 *>(bdst1 + bo + 128) = fp16_of_int8x8(make_uint2(xv1.z, xv1.w));
                    }
                }
            }
            // hand pair P to its MMA warp
            tmem_wait_st();
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(kBarMEmpty + st));   // this warp is done with input stage st
                mbar_arrive(bar(kBarABFull + sl));
            }
            if (++st == kStages) {
                st = 0;
                st_par ^= 1u;
            }
        }
    } else {
        // ---------------- folder warps: D read back and accumulated ----------------
        const int f = warp - kFolderWarp0;
        const int q = warp & 3, th = f >> 2;   // row quarter (the warp's tensor-memory lanes); tokens 32 th..+31
        const bool rows_q = q < ctiles;
        const int tile = blockIdx.x * ctiles + q;
        const bool tile_ok = rows_q && tile < tiles;
        const int row = tile * tgi::kTileRows + lane;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const bool epi = rows_q && 32 * th < M;   // warp-uniform: this warp's rows and tokens exist
        // int64 accumulators of tokens 32 th + j (j = 0..31) for this row: [token][row] layout, + 128 j
        int64_t *accs = reinterpret_cast<int64_t *>(smem + kOffAcc) + 32 * th * kRowsPerCta + 32 * q + lane;
        // this row's scale of group g: sc_row[32 g] (the blob's scales, 128 bytes per tile and group)
        const int32_t *sc_row = reinterpret_cast<const int32_t *>(scales) + (size_t)(tile_ok ? tile : 0) * G * 32 + lane;
        const uint32_t dbase = tmem + lane_off + kColD + 32u * (uint32_t)th;

        // D buffers start free
        __syncwarp();
        if (lane == 0)
            for (int db = 0; db < kDBufs; db++)
                mbar_arrive(bar(kBarDEmpty + db));

        uint32_t acc32[32];
#pragma unroll
        for (int j = 0; j < 32; j++)
            acc32[j] = 0;
        uint64_t dsum = 0;
        uint32_t dblk = 0;
        int nblk = 0;
        auto flush = [&]() {
            const uint32_t c = kOffsetBits * dblk;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                accs[128 * j] += (int64_t)(int32_t)(acc32[j] - c);
                acc32[j] = 0;
            }
            dblk = 0;
            nblk = 0;
        };
        // one group's 32 accumulator values (bit patterns 0x4B400000 + P once offset), scaled by dgp
        auto fold = [&](uint32_t (&v0)[16], uint32_t (&v1)[16], int dgp) {
#pragma unroll
            for (int j = 0; j < 16; j++) {
                v0[j] = __float_as_uint(__fadd_rn(__uint_as_float(v0[j]), 12582912.0f));
                v1[j] = __float_as_uint(__fadd_rn(__uint_as_float(v1[j]), 12582912.0f));
            }
            if (kNarrow) {
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    acc32[j] += v0[j] * (uint32_t)dgp;
                    acc32[16 + j] += v1[j] * (uint32_t)dgp;
                }
                dblk += (uint32_t)dgp;
                if (++nblk == kBlock)
                    flush();
            } else if (kFold == kFoldWide) {
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    accs[128 * j] = (int64_t)mad_wide(v0[j], dgp, (uint64_t)accs[128 * j]);
                    accs[128 * (16 + j)] = (int64_t)mad_wide(v1[j], dgp, (uint64_t)accs[128 * (16 + j)]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    accs[128 * j] += ((int64_t)(int32_t)(v0[j] - kOffsetBits) * dgp) >> frac;   // the group's floor
                    accs[128 * (16 + j)] += ((int64_t)(int32_t)(v1[j] - kOffsetBits) * dgp) >> frac;
                }
            }
        };
        auto scale_of = [&](int g) { return (tile_ok && g < G) ? __ldg(sc_row + (size_t)32 * g) : 0; };
        int dcur0 = scale_of(0), dcur1 = scale_of(1);
#pragma unroll 1
        for (int P = 0; P < npairs; P++) {
            const int sl = P & 1;
            const uint32_t par = (uint32_t)(P >> 1) & 1u;
            const int ng = min(kPair, G - kPair * P);
            // the next pair's scales load while this pair is read back
            const int dn0 = scale_of(kPair * (P + 1)), dn1 = scale_of(kPair * (P + 1) + 1);
            wait(kBarDFull + sl, par);
            fence_after_sync();
            const uint32_t dcol = dbase + (uint32_t)(kPair * kMaxN * sl);
            uint32_t v0[16], v1[16];
            if (epi) {
                tmem_ld16(dcol, v0);
                tmem_ld16(dcol + 16u, v1);
                tmem_wait_ld(v0);
                tmem_wait_ld(v1);
                fold(v0, v1, dcur0);
            }
            if (ng > 1 && epi) {
                tmem_ld16(dcol + kMaxN, v0);
                tmem_ld16(dcol + kMaxN + 16u, v1);
                tmem_wait_ld(v0);
                tmem_wait_ld(v1);
            }
            // D buffer sl read back: free for pair P + 2
            fence_before_sync();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(bar(kBarDEmpty + sl));
            if (ng > 1 && epi)
                fold(v0, v1, dcur1);
            dsum += (uint64_t)(int64_t)dcur0 + (uint64_t)(int64_t)dcur1;
            dcur0 = dn0;
            dcur1 = dn1;
        }
        if (kNarrow && epi)
            flush();
        // wide fold: y[m][r] = acc_m - 0x4B400000 * sum_g d (mod 2^64); otherwise acc_m
        if (epi && tile_ok && row < N) {
            const uint64_t corr = kFold == kFoldWide ? (uint64_t)kOffsetBits * dsum : 0ull;
#pragma unroll
            for (int j = 0; j < 32; j++) {
                const int m = 32 * th + j;
                if (m < M)
                    y[(size_t)m * N + row] = (int64_t)((uint64_t)accs[128 * j] - corr);
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        fence_after_sync();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace

namespace tgi {

int gemv_i8_mma(const uint4 *masks, const int32_t *scales, const int8_t *x, int64_t *y, int N, int G,
                int tiles, int M, int64_t max_abs_scale, bool q1, int frac, int64_t wait_cycles, cudaStream_t s)
{
    const long long wait_limit = wait_cycles > 0 ? (long long)wait_cycles : kDefaultWaitCycles;
    // cuTensorMapEncodeTiled from the driver, looked up once
    using encode_fn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
    static std::mutex mu;
    static encode_fn encode = nullptr;
    static uint64_t attr_set = 0;   // bit d: the kernels' shared-memory limit is raised on device d
    int dev = 0, nsm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TG_ERR_CUDA;
    const int fold = frac > 0 ? kFoldFloor : max_abs_scale <= kNarrowMaxScale ? kFoldNarrow : kFoldWide;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!encode) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn)
                return TG_ERR_CUDA;
            encode = reinterpret_cast<encode_fn>(fn);
        }
        const uint64_t dev_bit = dev < 64 ? 1ull << dev : 0ull;   // (devices past 64: set every call)
        if (!(attr_set & dev_bit)) {
            void (*kernels[6])(const unsigned char *, const unsigned char *, const CUtensorMap, int64_t *, int, int,
                               int, int, int, int, long long) = {
                gemv_i8_mma_kernel<false, kFoldNarrow>, gemv_i8_mma_kernel<false, kFoldWide>,
                gemv_i8_mma_kernel<false, kFoldFloor>,  gemv_i8_mma_kernel<true, kFoldNarrow>,
                gemv_i8_mma_kernel<true, kFoldWide>,    gemv_i8_mma_kernel<true, kFoldFloor>};
            for (auto k : kernels)
                if (cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) != cudaSuccess)
                    return TG_ERR_CUDA;
            attr_set |= dev_bit;
        }
    }
    // x as a 2D tensor [M rows][K bytes]; boxes of 64 rows x 128 bytes, 128-byte swizzle
    CUtensorMap xmap;
    const cuuint64_t dims[2] = {(cuuint64_t)G * TG_GROUP, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)G * TG_GROUP};
    const cuuint32_t box[2] = {TG_GROUP, kMaxN};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t *>(x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return TG_ERR_CUDA;
    // Tiles per CTA: the fewest that still fit every CTA in one wave (one CTA per SM),
    // so that a shape with fewer than 4 x #SMs tiles spreads over more SMs; a CTA's
    // per-group work shrinks with its tiles, the activation conversion does not.
    int ctiles = 4;
    for (int c = 1; c < 4; c++)
        if ((tiles + c - 1) / c <= nsm) {
            ctiles = c;
            break;
        }
    const int grid = (tiles + ctiles - 1) / ctiles;
    const auto *mk = reinterpret_cast<const unsigned char *>(masks);
    const auto *sc = reinterpret_cast<const unsigned char *>(scales);
#define TGI_MMA_LAUNCH(Q, F) \
    gemv_i8_mma_kernel<Q, F><<<grid, kThreads, kSmemBytes, s>>>(mk, sc, xmap, y, N, G, tiles, M, frac, ctiles, \
                                                               wait_limit)
    if (q1) {
        if (fold == kFoldNarrow)
            TGI_MMA_LAUNCH(true, kFoldNarrow);
        else if (fold == kFoldWide)
            TGI_MMA_LAUNCH(true, kFoldWide);
        else
            TGI_MMA_LAUNCH(true, kFoldFloor);
    } else {
        if (fold == kFoldNarrow)
            TGI_MMA_LAUNCH(false, kFoldNarrow);
        else if (fold == kFoldWide)
            TGI_MMA_LAUNCH(false, kFoldWide);
        else
            TGI_MMA_LAUNCH(false, kFoldFloor);
    }
#undef TGI_MMA_LAUNCH
    return cudaGetLastError() == cudaSuccess ? TG_OK : TG_ERR_CUDA;
}

}  // namespace tgi
