// vca_device.cuh -- inline-PTX building blocks for sm_103a (Blackwell Ultra):
// mbarriers with bounded waits, TMA tile loads, tcgen05 MMA / TMEM access,
// shared-memory matrix descriptors, and the number-format helpers the
// VC-Attention kernels share.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>

namespace vca {

constexpr int kBlk = 128;   // the 128-token hardware block (tile edge)
constexpr int kD = 128;     // head width

// Status codes written to the device status word (mirror vca_status).
constexpr int kErrTimeout = 4;

// ---------------------------------------------------------------------------
// Addresses and time
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// try_wait that may suspend the thread (up to `hint_ns`) until the phase
// completes, instead of returning at once: waiting warps then stop competing
// for issue slots with the warps doing the work.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed, or give
// up: after `limit_ns` of wall time, or as soon as another thread of the CTA
// has raised `*abort`.  Returns false on giving up (and raises *abort).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int *abort, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*reinterpret_cast<volatile int *>(abort)) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *reinterpret_cast<volatile int *>(abort) = 1;
            return false;
        }
    }
}

// mbar_wait for a waiter on the critical path: polls without suspending (a
// suspended thread resumes some hundreds of cycles after the phase
// completes), with the same give-up rules.  Each poll is one shared-memory
// round trip, so the spinning thread takes few issue slots from its
// neighbours.
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity, int *abort, uint64_t limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_test_wait(bar, parity)) return true;
        if (*reinterpret_cast<volatile int *>(abort)) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            *reinterpret_cast<volatile int *>(abort) = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------------------
// Proxy fences
// ---------------------------------------------------------------------------
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor-core operand reads, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// TMA (bulk tensor copies global -> shared, completion via mbarrier tx count)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const void *tmap, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing on `bar` through its transaction count.
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(smem_dst)),
                 "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, TMEM loads/stores, fences
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Arrive on `bar` once every tcgen05 operation this thread issued so far is done.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// D(tmem, fp32) (+)= A(smem) * B(smem)^T, FP8/FP6/FP4 operands.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem, fp32) (+)= A(tmem) * B(smem)^T, FP8/FP6/FP4 operands: A holds M rows
// in TMEM lanes and K along columns, four 8-bit elements per 32-bit column.
__device__ __forceinline__ void mma_f8f6f4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem, fp32) (+)= A(tmem) * B(smem)^T, 16-bit operands: A holds M rows in
// TMEM lanes and K along columns, two 16-bit elements per 32-bit column (the
// lower K index in the low half).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D(tmem, fp32) (+)= A(smem) * B(smem)^T, 16-bit operands.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Instruction descriptor (dense, fp32 accumulator, operands K-major unless
// flagged).
// atype/btype: kind::f8f6f4 -> 0 = E4M3; kind::f16 -> 0 = F16, 1 = BF16.
// a_mn / b_mn: the operand is MN-major instead (16-bit types only).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, uint32_t atype, uint32_t btype, uint32_t a_mn = 0,
                                                  uint32_t b_mn = 0) {
    return (1u << 4)                                   // D format: fp32
           | (atype << 7) | (btype << 10)              // A, B formats
           | (a_mn << 15) | (b_mn << 16)               // A, B major-ness
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms of 1024 bytes (the layout a
// TMA SWIZZLE_128B load produces).  The atom base must be 1024-byte aligned;
// stepping K inside the atom advances the start address by the slice's bytes.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;            // stride byte offset: next 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                    // 128-byte swizzle
    return d;
}

// Shared-memory matrix descriptor for a K-major operand with the 64-byte
// swizzle, as a TMA load with CU_TENSOR_MAP_SWIZZLE_64B writes it: rows of 64
// bytes, 8-row atoms of 512 bytes one after another (the tile 512-byte
// aligned).  A K step inside the row is a start-address step (16-byte units).
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address
    d |= static_cast<uint64_t>(1) << 16;                    // leading byte offset (unused here)
    d |= static_cast<uint64_t>(512 >> 4) << 32;             // stride byte offset: next 8-row atom
    d |= static_cast<uint64_t>(1) << 46;                    // descriptor version for tcgen05
    d |= static_cast<uint64_t>(4) << 61;                    // 64-byte swizzle
    return d;
}

// Shared-memory matrix descriptor for an MN-major 16-bit operand with the
// 128-byte swizzle: rows are K indices, each row holds 64 consecutive M (or N)
// elements (128 bytes), 8-row atoms of 1024 bytes follow each other along K
// (stride byte offset), and the next 64 M/N elements start `panel_bytes`
// further on (leading byte offset).  Stepping K by 16 advances the start
// address by 16 rows (2048 bytes).
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t panel_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);            // start address
    d |= static_cast<uint64_t>((panel_bytes >> 4) & 0x3FFFu) << 16;  // leading byte offset: next MN panel
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                     // stride byte offset: next 8 K rows
    d |= static_cast<uint64_t>(1) << 46;                             // descriptor version for tcgen05
    d |= static_cast<uint64_t>(2) << 61;                             // 128-byte swizzle
    return d;
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled tile.
__device__ __forceinline__ uint32_t sw128_offset(uint32_t row, uint32_t chunk) {
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

#define VCA_TMEM_LD32(taddr, r)                                                                                   \
    asm volatile(                                                                                                 \
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"   \
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"                                        \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),   \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), \
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])  \
        : "r"(taddr))

// tcgen05.ld of 32 (16) columns that also returns `m`, the largest of the
// thread's loaded values as fp32 (NaN ignored, as max.f32 does): sm_103a's
// reducing TMEM load, measured on the hardware to return the data unchanged.
#define VCA_TMEM_LDMAX32(taddr, r, m)                                                                             \
    asm volatile(                                                                                                 \
        "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"   \
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"                           \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),   \
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), \
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), \
          "=f"(m)                                                                                                 \
        : "r"(taddr))

#define VCA_TMEM_LDMAX16(taddr, r, m)                                                                             \
    asm volatile(                                                                                                 \
        "tcgen05.ld.red.sync.aligned.32x32b.x16.max.f32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, " \
        "%16, [%17];"                                                                                             \
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),         \
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),   \
          "=f"(m)                                                                                                 \
        : "r"(taddr))

#define VCA_TMEM_ST32(taddr, r)                                                                                   \
    asm volatile(                                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"    \
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),                         \
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),        \
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),           \
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),          \
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])                       \
        : "memory")

#define VCA_TMEM_ST16(taddr, r)                                                                                   \
    asm volatile(                                                                                                 \
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"  \
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),    \
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])             \
        : "memory")

#define VCA_TMEM_ST8(taddr, r)                                                                                    \
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),    \
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])                         \
                 : "memory")

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Number formats
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) { return __uint_as_float(static_cast<uint32_t>(h) << 16); }

// Two fp32 values -> two bf16 (round to nearest even); `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// hi + lo split of two values for bf16 operands, packed: h = bf16(a) |
// bf16(b) << 16 and l = bf16(a - hi(a)) | bf16(b - hi(b)) << 16, with
// hi(x) = bf16(x) (x - hi(x) is exact in fp32; bf16 of it keeps x to ~16
// significant bits).  One conversion per word; the hi halves are read back as
// fp32 by placing them in the high 16 bits.
__device__ __forceinline__ void split_pack_bf16x2(float a, float b, uint32_t &h, uint32_t &l) {
    h = pack_bf16x2(a, b);
    const float ha = __uint_as_float(h << 16), hb = __uint_as_float(h & 0xffff0000u);
    l = pack_bf16x2(__fsub_rn(a, ha), __fsub_rn(b, hb));
}


// Four fp32 values -> four E4M3 bytes of one word (byte i = value i; round to
// nearest even, saturate to 448): two cvt instructions and a register pack.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    uint32_t w;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(w)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return w;
}

__device__ __forceinline__ uint32_t e4m3(float x) {
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}

// Eight fp32 values -> eight E2M1 codes in one word (value i in nibble i;
// round to nearest even, saturate to 6): four cvt instructions and a pack.
__device__ __forceinline__ uint32_t e2m1x8(const float (&v)[8]) {
    uint32_t w;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(w)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return w;
}

// Value of an E4M3 byte (exact in fp32).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(code), __NV_E4M3);
    return __half2float(__half(h));
}

// ExpCast-FP8: the E4M3 byte of p = 2^(s - m) from the raw score with one FMA.
//   t = fma(s_raw, 8c, 55.65 - 8m)  (c8 = 8c and bias = 55.65 - 8m precomputed)
//   code = rne(t); code < 8 -> 0 (below the normal range); code > 126 -> 126.
// Adding 1.5 * 2^23 rounds t to an integer (nearest even) in the float's low
// mantissa bits, so the code is the low byte of the sum's bit pattern.
constexpr float kExpcastOffset = 55.65f;     // 56 + beta, beta = -0.35
constexpr float kMagic = 12582912.0f;        // 1.5 * 2^23

// Packed fp32 pairs: two lanes per instruction on sm_100 and later.
__device__ __forceinline__ uint64_t pk2(uint32_t lo, uint32_t hi) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "r"(lo), "r"(hi));
    return d;
}
__device__ __forceinline__ void upk2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// Byte permute with the selector's sign-replication bit honoured.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Four ExpCast codes packed in one word (byte i = element i).  Per element one
// saturating fp32 FMA forms u = t / 256 clamped to [0, 1]: with c8s = 8c / 256
// and bs = (55.65 - 8m) / 256 (both exact, a power-of-two scaling), u is
// fma(s, 8c, 55.65 - 8m) / 256 with the same single rounding, and negative t
// and NaN give 0.  Adding 1.5 * 2^15 (ulp 2^-8, packed two per instruction)
// rounds 256 u = t to an integer, nearest even, in the low mantissa bits: the
// pattern is 0x47400000 + code.  kClip caps u at 126/256 (codes above 126
// become 126).  The codes are packed with one PRMT for codes 0 and 1 (over the
// pattern's zero byte 1) and integer multiply-adds for codes 2 and 3 (the
// 0x4740 high half vanishes times 2^16 or 2^24, modulo 2^32), and the bytes
// 1..7 are zeroed together: a byte b <= 126 is >= 8 exactly when b + 120 has
// its top bit set, which PRMT replicates into a byte mask.  Without kClip the
// caller guarantees codes <= 126: that holds when fp32(s * c) <= fp32(m + 8)
// and |m| < 2^22, because t then exceeds 55.65 by at most 8 * 8 + 16 ulp(m)
// <= 68.
constexpr float kExpcastFastMax = 4194304.0f;   // 2^22
constexpr float kMagicSat = 49152.0f;           // 1.5 * 2^15
// `one` must hold 1: it turns the flush's integer add into a multiply-add,
// which issues to the FMA pipe instead of the ALU pipe (the caller passes a
// value the compiler cannot fold, e.g. a kernel parameter).
template <bool kClip>
__device__ __forceinline__ uint32_t expcast4(const uint32_t (&s)[4], float c8s, float bs, uint32_t one) {
    float u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        asm("fma.rn.sat.f32 %0, %1, %2, %3;" : "=f"(u[e]) : "f"(__uint_as_float(s[e])), "f"(c8s), "f"(bs));
        if (kClip) u[e] = fminf(u[e], 126.0f / 256.0f);
    }
    const uint64_t magic2 = pk2(__float_as_uint(kMagicSat), __float_as_uint(kMagicSat));
    float x[4];
    upk2(add2(pk2(__float_as_uint(u[0]), __float_as_uint(u[1])), magic2), x[0], x[1]);
    upk2(add2(pk2(__float_as_uint(u[2]), __float_as_uint(u[3])), magic2), x[2], x[3]);
    uint32_t w = prmt(__float_as_uint(x[0]), __float_as_uint(x[1]), 0x1140);
    asm("mad.lo.u32 %0, %1, 65536, %0;" : "+r"(w) : "r"(__float_as_uint(x[2])));
    asm("mad.lo.u32 %0, %1, 16777216, %0;" : "+r"(w) : "r"(__float_as_uint(x[3])));
    uint32_t t;
    asm("mad.lo.u32 %0, %1, %2, 2021161080;" : "=r"(t) : "r"(w), "r"(one));   // w + 0x78787878
    return w & prmt(t, 0u, 0xBA98);
}

// Two fp32 products, each rounded to nearest even (one packed instruction).
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Four ExpCast codes packed in one word (byte i = element i) when every code
// is at most 126 (|m| < 2^22 and fp32(s c) <= fp32(m + 8), as for expcast4<false>),
// in nine instructions:
//   t = fma(s, 8c, 55.65 - 8m)            two packed FMAs (t with its one rounding)
//   y = t * 2^-149                         two packed multiplies: the exact product
//       rounds, nearest even, to a multiple of the smallest subnormal, so y's
//       bit pattern is rne(t) for 0 <= t < 2^23, and a negative t leaves the
//       sign bit set (a negative 32-bit integer)
//   cvt.pack.sat.u8.s32.b32 twice         clamps each pattern to [0, 255] as a
//       signed integer and packs it: d = (c & 0xffff) << 16 | sat(a) << 8 | sat(b)
//       (the layout measured on the device)
//   the flush of codes 1..7 as in expcast4.
// Subnormal results are kept: neither the multiply nor the FMA flushes to zero.
__device__ __forceinline__ uint32_t expcast4_fast(const uint32_t (&s)[4], uint64_t c8x2, uint64_t bx2, uint32_t one) {
    const uint64_t tiny2 = pk2(1u, 1u);   // 2^-149 in both halves
    const uint64_t y01 = mul2(fma2(pk2(s[0], s[1]), c8x2, bx2), tiny2);
    const uint64_t y23 = mul2(fma2(pk2(s[2], s[3]), c8x2, bx2), tiny2);
    uint32_t y[4];
    asm("mov.b64 {%0, %1}, %2;" : "=r"(y[0]), "=r"(y[1]) : "l"(y01));
    asm("mov.b64 {%0, %1}, %2;" : "=r"(y[2]), "=r"(y[3]) : "l"(y23));
    uint32_t hi, w;
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(y[3]), "r"(y[2]), "r"(0u));
    asm("cvt.pack.sat.u8.s32.b32 %0, %1, %2, %3;" : "=r"(w) : "r"(y[1]), "r"(y[0]), "r"(hi));
    uint32_t t;
    asm("mad.lo.u32 %0, %1, %2, 2021161080;" : "=r"(t) : "r"(w), "r"(one));   // w + 0x78787878
    return w & prmt(t, 0u, 0xBA98);
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------------------
// Host: the driver's tensor-map encoder, looked up through the runtime (no
// link against libcuda)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

}  // namespace vca
