// Device building blocks of the W12 kernels (sm_103a): mbarrier / TMA /
// tcgen05 wrappers in inline PTX, and the in-register W12 decode.
//
// Register decode ("decoded inside the GEMM registers": "SpecPilot: an agent
// doubled speculative decoding speed, and the 10.87x needs context", §The
// mechanisms it found; "decodes bit-exactly inside the GEMM":
// "StargazerX0/SpecPilot", §What it is).  One thread owns one row of a
// 32-column chunk and turns its 48 packed bytes into 16 words of BF16 pairs:
//
//   exponent lookup  PRMT selects bytes with a 4-bit selector whose top bit
//                    means "replicate the sign of the selected byte".  With
//                    the table in four words R0..R3 (slots 0-15) and
//                    R0' = R0 ^ signs(R2), R1' = R1 ^ signs(R3):
//                      e = prmt(R0', R1', c) ^ prmt(R2, R3, c ^ 8)
//                    gives T[c] for every c < 15, because the format keeps
//                    slots j and j + 8 on the same top bit.  2 PRMT + 1 XOR
//                    per four weights (plus selector prep per eight).
//   assembly         prmt(S, E) interleaves [E1 S1 E0 S0]; since each S byte
//                    is (mantissa << 1) | partner's sign, one 32-bit rotate
//                    right by 1 lands both signs, exponents and mantissas on
//                    their BF16 bits: 1 PRMT + 1 SHF per two weights.
//   escapes          code 15: the exponent byte is patched from the escape
//                    list (flags by a carry trick, warp scan for offsets).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace w12 {
namespace dev {

// ---------------------------------------------------------------- basics
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// PRMT in its default mode: selector nibble bits 0-2 pick a byte of {b, a},
// bit 3 replaces it by its sign replicated over 8 bits.  (Written in PTX
// because __byte_perm is documented to use 3-bit selectors only.)
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ uint32_t rotr1(uint32_t x) { return __funnelshift_r(x, x, 1); }

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// 16-byte shared-memory load through a 32-bit shared address.
__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(saddr));
    return v;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Add to the expected transaction bytes of the current phase without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test: true when the phase with `parity` has completed (never
// waits, unlike try_wait).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// As above, but a thread whose phase is not complete may sleep in hardware
// for up to `hint_ns` (it wakes as soon as the phase completes).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Bounded wait: true once the phase with `parity` has completed, false when
// `deadline_ns` (globaltimer) passes first.  Nothing here can spin forever.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t deadline_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if ((i & 7u) == 0 && globaltimer_ns() > deadline_ns) return false;
    }
}

// ---------------------------------------------------------------- TMA
// 1-D bulk copy global -> shared, completion counted in bytes on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policy for data read once (the weight stream): its lines are the first
// to go, so that small data read again later (x, split-K partial sums, segment
// headers) stays in L2.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// As bulk_g2s, with an L2 cache policy.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// 2-D tiled tensor copy global -> shared (coordinates in elements, x first).
__device__ __forceinline__ void tma_load_2d(void *dst, const void *tmap, int32_t x, int32_t y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(dst)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start
// launching, and wait until the previous one has completed and its writes are
// visible.
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Warm L2 with `bytes` (a multiple of 16) from a 16-byte aligned address.
__device__ __forceinline__ void prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// ---------------------------------------------------------------- tcgen05
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
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16 (BF16 in, fp32 accumulate).
__device__ __forceinline__ void mma_tmem_a(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
        "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T.
__device__ __forceinline__ void mma_smem_a(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_taddr),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on `bar` once every tcgen05 operation this thread issued has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// Warp-collective store of 16 32-bit columns (lane i -> TMEM lane base + i).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr), "r"(v[0]),
        "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warp-collective load of 16 32-bit columns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Make generic-proxy writes to shared memory visible to the async proxy
// (tensor cores reading an operand written by st.shared).
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor (tcgen05): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1 at bit 46, and the
// layout type in bits 61-63 (0 none, 2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(layout & 7u) << 61;
    return d;
}

// Instruction descriptor, kind::f16: fp32 D, BF16 A and B, both K-major,
// N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t m, uint32_t n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

// ---------------------------------------------------------------- W12 decode
// The segment table in the four words the lookup uses (see the file header).
struct Table {
    uint32_t u0, u1, u2, u3;
};

__device__ __forceinline__ Table make_table(uint4 t) {
    Table r;
    r.u0 = t.x ^ prmt(t.z, 0u, 0xBA98u);  // xor with the signs of slots 8..11
    r.u1 = t.y ^ prmt(t.w, 0u, 0xBA98u);  // xor with the signs of slots 12..15
    r.u2 = t.z;
    r.u3 = t.w;
    return r;
}

// Exponent bytes of the eight weights whose codes fill word w (code k in
// nibble k): ea gets codes 0-3, eb codes 4-7, one exponent per byte.
__device__ __forceinline__ void lookup8(const Table &T, uint32_t w, uint32_t &ea, uint32_t &eb) {
    const uint32_t wh = w >> 16;
    ea = prmt(T.u0, T.u1, w) ^ prmt(T.u2, T.u3, w ^ 0x8888u);
    eb = prmt(T.u0, T.u1, wh) ^ prmt(T.u2, T.u3, wh ^ 0x8888u);
}

// E[j] = exponents of columns 4j..4j+3 of the thread's row.
__device__ __forceinline__ void decode_exponents(const Table &T, const uint4 &codes, uint32_t (&E)[8]) {
    lookup8(T, codes.x, E[0], E[1]);
    lookup8(T, codes.y, E[2], E[3]);
    lookup8(T, codes.z, E[4], E[5]);
    lookup8(T, codes.w, E[6], E[7]);
}

// out[i] = BF16 pair (column 2i in the low half, 2i+1 in the high half).
__device__ __forceinline__ void assemble(const uint4 &s_lo, const uint4 &s_hi, const uint32_t (&E)[8],
                                         uint32_t (&out)[16]) {
    const uint32_t S[8] = {s_lo.x, s_lo.y, s_lo.z, s_lo.w, s_hi.x, s_hi.y, s_hi.z, s_hi.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        out[2 * j] = rotr1(prmt(S[j], E[j], 0x5140u));      // [E1 S1 E0 S0]
        out[2 * j + 1] = rotr1(prmt(S[j], E[j], 0x7362u));  // [E3 S3 E2 S2]
    }
}

// Bit 4p+3 set exactly where nibble p of w equals 15 (the escape code):
// adding 7 to the low three bits of ~w carries into bit 3 unless they are 0.
__device__ __forceinline__ uint32_t escape_flags(uint32_t w) {
    const uint32_t t = (~w & 0x77777777u) + 0x77777777u;
    return ~t & w & 0x88888888u;
}

// Patch the escaped exponents of one thread's row chunk, reading the escape
// bytes in column order from src.
__device__ __forceinline__ void patch_escapes(const uint32_t (&f)[4], const uint8_t *src, uint32_t (&E)[8]) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t fj = (f[j >> 1] >> (16 * (j & 1))) & 0x8888u;
        while (fj) {
            const uint32_t b = (uint32_t)__ffs(fj) - 1u;  // 3, 7, 11 or 15
            fj &= fj - 1u;
            const uint32_t sh = (b >> 2) << 3;
            const uint32_t e = *src++;
            E[j] = (E[j] & ~(0xFFu << sh)) | (e << sh);
        }
    }
}

// Warp-wide escape step for one quarter-chunk: every lane finds its escapes,
// an exclusive prefix over the lanes gives each lane its first byte in the
// quarter's run (rows in lane order, columns in order), and the exponents are
// patched.  Returns the warp's escape count (to advance the run).  When few
// lanes hold escapes (the common case) the prefix is gathered from those lanes
// only; otherwise a shuffle scan runs.
__device__ __forceinline__ uint32_t warp_escapes(const uint4 &codes, const uint8_t *run, uint32_t (&E)[8]) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t f[4] = {escape_flags(codes.x), escape_flags(codes.y), escape_flags(codes.z),
                           escape_flags(codes.w)};
    const uint32_t cnt = __popc(f[0]) + __popc(f[1]) + __popc(f[2]) + __popc(f[3]);
    const uint32_t holders = __ballot_sync(0xFFFFFFFFu, cnt != 0);
    uint32_t excl = 0, total = 0;
    if (__popc(holders) <= 4) {
        uint32_t h = holders;
        while (h) {
            const uint32_t l = (uint32_t)__ffs(h) - 1u;
            h &= h - 1u;
            const uint32_t c = __shfl_sync(0xFFFFFFFFu, cnt, l);
            total += c;
            if (l < lane) excl += c;
        }
    } else {
        uint32_t incl = cnt;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
            if (lane >= (uint32_t)d) incl += v;
        }
        total = __shfl_sync(0xFFFFFFFFu, incl, 31);
        excl = incl - cnt;
    }
    if (cnt) patch_escapes(f, run + excl, E);
    return total;
}

// ---- half-chunk forms: one thread, one row, 16 columns (half h of a chunk)

// E[j] = exponents of columns 16h + 4j .. 16h + 4j + 3 (codes in words w0, w1).
__device__ __forceinline__ void decode_exponents_half(const Table &T, uint32_t w0, uint32_t w1, uint32_t (&E)[4]) {
    lookup8(T, w0, E[0], E[1]);
    lookup8(T, w1, E[2], E[3]);
}

// out[i] = BF16 pair of columns 16h + 2i, 16h + 2i + 1.
__device__ __forceinline__ void assemble_half(const uint4 &s, const uint32_t (&E)[4], uint32_t (&out)[8]) {
    const uint32_t S[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        out[2 * j] = rotr1(prmt(S[j], E[j], 0x5140u));
        out[2 * j + 1] = rotr1(prmt(S[j], E[j], 0x7362u));
    }
}

// Two escape-free chunks of this thread's row: chunk a into va (16 words of
// BF16 pairs), chunk b into vb.
__device__ __forceinline__ void decode_pair_plain(const Table &T, const uint4 &a0, const uint4 &a1,
                                                  const uint4 &acd, const uint4 &b0, const uint4 &b1,
                                                  const uint4 &bcd, uint32_t (&va)[16], uint32_t (&vb)[16]) {
    uint32_t Ea0[4], Ea1[4], Eb0[4], Eb1[4];
    decode_exponents_half(T, acd.x, acd.y, Ea0);
    decode_exponents_half(T, acd.z, acd.w, Ea1);
    decode_exponents_half(T, bcd.x, bcd.y, Eb0);
    decode_exponents_half(T, bcd.z, bcd.w, Eb1);
    const uint32_t Sa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t Sb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const uint32_t ea = j < 4 ? Ea0[j & 3] : Ea1[j & 3];
        const uint32_t eb = j < 4 ? Eb0[j & 3] : Eb1[j & 3];
        va[2 * j] = rotr1(prmt(Sa[j], ea, 0x5140u));
        va[2 * j + 1] = rotr1(prmt(Sa[j], ea, 0x7362u));
        vb[2 * j] = rotr1(prmt(Sb[j], eb, 0x5140u));
        vb[2 * j + 1] = rotr1(prmt(Sb[j], eb, 0x7362u));
    }
}

// Exclusive prefix over the lanes of `cnt` and the warp total.  When no lane
// holds more than one escape (the common case) a ballot gives both; else a
// shuffle scan.
__device__ __forceinline__ void lane_prefix(uint32_t cnt, uint32_t &excl, uint32_t &total) {
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t holders = __ballot_sync(0xFFFFFFFFu, cnt != 0);
    if (__all_sync(0xFFFFFFFFu, cnt <= 1u)) {
        excl = __popc(holders & ((1u << lane) - 1u));
        total = __popc(holders);
        return;
    }
    uint32_t incl = cnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
        if (lane >= (uint32_t)d) incl += v;
    }
    total = __shfl_sync(0xFFFFFFFFu, incl, 31);
    excl = incl - cnt;
}

// Patch escaped exponents into E[0..3] (16 columns) from src, in column
// order, with a warp-uniform loop and predicated selects (no divergent
// branches): fh[0], fh[1] are the escape flags of the 16 columns.
__device__ __forceinline__ void patch_half(uint32_t f0, uint32_t f1, const uint8_t *src, uint32_t (&E)[4]) {
    const uint32_t mine = __popc(f0) + __popc(f1);
    const uint32_t rounds = __reduce_max_sync(0xFFFFFFFFu, mine);
    for (uint32_t t = 0; t < rounds; ++t) {
        const bool have = t < mine;
        const bool lo = f0 != 0u;
        const uint32_t fw = lo ? f0 : f1;
        const uint32_t b = (uint32_t)__ffs(fw) - 1u;    // 4p + 3 within the word
        const uint32_t k = (lo ? 0u : 8u) + (b >> 2);    // column 0..15
        const uint32_t clear = fw & (fw - 1u);
        f0 = lo ? clear : f0;
        f1 = lo ? f1 : clear;
        const uint32_t e = have ? (uint32_t)src[t] : 0u;
        const uint32_t sh = (k & 3u) << 3;
        const uint32_t j = k >> 2;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const uint32_t patched = (E[jj] & ~(0xFFu << sh)) | (e << sh);
            E[jj] = (have && j == (uint32_t)jj) ? patched : E[jj];
        }
    }
}

// Escape step for 16 columns of a quarter-chunk row, before the exponent
// lookup: w0, w1 are their code words, fh0, fh1 their escape flags and src
// their first escape byte.  Common case: no lane holds more than one escape in
// its 16 columns.  Then a lane with one escape puts that exponent into slot 15
// of its own copy of the table, and the ordinary lookup decodes it.  Slot 15
// is looked up as sign(slot 7) ^ slot 15, and slot 7 as slot 7 ^ sign(slot
// 15), so this holds when the escaped exponent has the same top bit as T[7],
// or when the lane has no code 7 to get wrong.  Otherwise the exponents are
// patched after the lookup.  Warp-uniform control flow.
__device__ __forceinline__ void decode_exponents_16_esc(const Table &T, uint32_t w0, uint32_t w1, uint32_t fh0,
                                                        uint32_t fh1, const uint8_t *src, uint32_t (&E)[4]) {
    const uint32_t mine = __popc(fh0) + __popc(fh1);
    Table Tl = T;
    bool ok = mine <= 1u;
    if (mine == 1u) {
        const uint32_t e = *src;
        const uint32_t sign7 = (T.u1 & 0x80000000u) ? 0xFFu : 0u;  // top bit of slot 7
        // a top-bit mismatch only breaks code 7, which is harmless when none of
        // these 16 codes is 7 (code ^ 8 == 15)
        const bool no_code7 = (escape_flags(w0 ^ 0x88888888u) | escape_flags(w1 ^ 0x88888888u)) == 0u;
        ok = ((e ^ sign7) & 0x80u) == 0u || no_code7;
        Tl.u3 = (T.u3 & 0x00FFFFFFu) | ((e ^ sign7) << 24);
    }
    if (__all_sync(0xFFFFFFFFu, ok)) {
        decode_exponents_half(Tl, w0, w1, E);
    } else {
        decode_exponents_half(T, w0, w1, E);
        patch_half(fh0, fh1, src, E);
    }
}

// Half h of a quarter-chunk with escapes.  The escape run orders a row's 32
// columns together, so the lane prefix is taken over whole-row counts and the
// second half starts after the row's first-half escapes.  Returns the warp's
// escape count over the whole chunk (to advance the run).
__device__ __forceinline__ uint32_t decode_exponents_half_esc(const Table &T, const uint4 &codes, int h,
                                                             const uint8_t *run, uint32_t (&E)[4]) {
    const uint32_t f[4] = {escape_flags(codes.x), escape_flags(codes.y), escape_flags(codes.z),
                           escape_flags(codes.w)};
    const uint32_t c0 = __popc(f[0]) + __popc(f[1]);
    const uint32_t cnt = c0 + __popc(f[2]) + __popc(f[3]);
    uint32_t excl, total;
    lane_prefix(cnt, excl, total);
    decode_exponents_16_esc(T, h ? codes.z : codes.x, h ? codes.w : codes.y, h ? f[2] : f[0], h ? f[3] : f[1],
                            run + excl + (h ? c0 : 0u), E);
    return total;
}

// Both halves of a quarter-chunk with escapes, sharing one lane prefix.
// Returns the warp's escape count over the chunk.
__device__ __forceinline__ uint32_t decode_exponents_chunk_esc(const Table &T, const uint4 &codes,
                                                              const uint8_t *run, uint32_t (&E0)[4],
                                                              uint32_t (&E1)[4]) {
    const uint32_t f[4] = {escape_flags(codes.x), escape_flags(codes.y), escape_flags(codes.z),
                           escape_flags(codes.w)};
    const uint32_t c0 = __popc(f[0]) + __popc(f[1]);
    const uint32_t cnt = c0 + __popc(f[2]) + __popc(f[3]);
    uint32_t excl, total;
    lane_prefix(cnt, excl, total);
    decode_exponents_16_esc(T, codes.x, codes.y, f[0], f[1], run + excl, E0);
    decode_exponents_16_esc(T, codes.z, codes.w, f[2], f[3], run + excl + c0, E1);
    return total;
}

// Escapes of one quarter-chunk, patched after a plain decode: the ordinary
// lookup has given every escaped weight (code 15) a wrong exponent and the
// right sign and mantissa (both come from the S byte), so only its exponent
// field is replaced, from the escape run in row then column order: lane l's
// bytes start after the escapes of lanes 0..l-1 (a ballot prefix), and within
// the row they follow the columns.  w[i] holds the BF16 pair of columns 2i
// (low half) and 2i + 1 (high half); code word k of cd holds columns 8k..8k+7,
// one per nibble.  Returns the warp's escape count (to advance the run).
// Only lanes that hold escapes enter the patch loop.
__device__ __forceinline__ uint32_t patch_chunk_escapes(const uint4 &cd, const uint8_t *run, uint32_t (&w)[16]) {
    const uint32_t f[4] = {escape_flags(cd.x), escape_flags(cd.y), escape_flags(cd.z), escape_flags(cd.w)};
    const uint32_t cnt = __popc(f[0]) + __popc(f[1]) + __popc(f[2]) + __popc(f[3]);
    uint32_t excl, total;
    lane_prefix(cnt, excl, total);
    if (cnt != 0u) {
        const uint8_t *src = run + excl;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            uint32_t fk = f[k];
            while (fk != 0u) {
                const uint32_t p = ((uint32_t)__ffs(fk) - 1u) >> 2;  // column 8k + p
                fk &= fk - 1u;
                const uint32_t sh = (p & 1u) ? 23u : 7u;             // exponent field of the high or low half
                const uint32_t keep = ~(0xFFu << sh), e = (uint32_t)(*src++) << sh;
                const uint32_t word = p >> 1;                       // w[4k + word]
#pragma unroll
                for (int i = 0; i < 4; ++i) w[4 * k + i] = word == (uint32_t)i ? (w[4 * k + i] & keep) | e : w[4 * k + i];
            }
        }
    }
    return total;
}

// Arrive on an mbarrier once for the whole warp (after ordering every lane's
// earlier accesses), without a divergent branch.
__device__ __forceinline__ void warp_arrive(uint64_t *bar) {
    __syncwarp();
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "elect.sync _|p, 0xffffffff;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// Split-K arrival: add 1 to a tile's counter at GPU scope with acquire-release
// semantics and return the old value.  The release half publishes this
// thread's earlier stores and, cumulatively, those it has synchronised with
// (the CTA's partials, ordered before it by an mbarrier or __syncwarp); the
// acquire half lets the last arrival read every other CTA's partials.  One
// ordered atomic instead of a full fence on each side.
__device__ __forceinline__ uint32_t arrive_acq_rel(uint32_t *counter) {
    uint32_t old;
    asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// Hint: bring the 128-byte line holding `a` into this SM's L1 (no register
// is written; a later ld.global.ca of the line hits L1 if it is still there).
__device__ __forceinline__ void prefetch_l1(const void *a) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(a));
}

// Acquire load of a split-K counter at GPU scope: a value showing that the
// other CTAs of a tile have arrived also makes their partial sums visible.
__device__ __forceinline__ uint32_t load_acquire_gpu(const uint32_t *counter) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    return v;
}

// The same split into its parts, for a thread that arrives on several
// counters: one release fence, relaxed increments that are all in flight at
// once, and (when one of them was the last arrival) one acquire fence.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }
__device__ __forceinline__ uint32_t arrive_relaxed(uint32_t *counter) {
    uint32_t old;
    asm volatile("atom.add.relaxed.gpu.global.u32 %0, [%1], 1;" : "=r"(old) : "l"(counter) : "memory");
    return old;
}

// ---------------------------------------------------------------- Q8 copy
// 16 int8 weights (two's complement; one chunk half of a row) to 8 BF16 pairs,
// lower column in the low half, exactly: byte b ^ 0x80 = b + 128 goes into
// the low mantissa bits of 2^23 (0x4B000000), and subtracting 2^23 + 128 in
// fp32 leaves b; |b| <= 128 keeps the value exact in BF16, so its top 16 bits
// are the BF16 pattern.  The subtractions run two at a time (sub.f32x2).
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ void q8_half(const uint4 &v, uint32_t (&out)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    constexpr uint64_t kMagic2 = 0x4B0000804B000080ull;  // (2^23 + 128, 2^23 + 128)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t u = w[j] ^ 0x80808080u;
        const uint64_t p01 = ((uint64_t)prmt(u, 0x4B000000u, 0x7441u) << 32) | prmt(u, 0x4B000000u, 0x7440u);
        const uint64_t p23 = ((uint64_t)prmt(u, 0x4B000000u, 0x7443u) << 32) | prmt(u, 0x4B000000u, 0x7442u);
        const uint64_t d01 = sub_f32x2(p01, kMagic2), d23 = sub_f32x2(p23, kMagic2);
        out[2 * j] = prmt((uint32_t)d01, (uint32_t)(d01 >> 32), 0x7632u);
        out[2 * j + 1] = prmt((uint32_t)d23, (uint32_t)(d23 >> 32), 0x7632u);
    }
}

// ---------------------------------------------------------------- argmax
// LM-head argmax ("certified exact-argmax LM head": "SpecPilot: an agent
// doubled speculative decoding speed, and the 10.87x needs context", §The
// mechanisms it found).  A candidate (fp32 logit v of row n) becomes a 64-bit
// key whose unsigned order is: larger v first, then smaller n; the maximum
// key over all rows is the argmax with ties to the lowest index.  -0 ranks as
// +0 and NaN as -inf.  Key 0 is below every real candidate.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t n) {
    uint32_t b = __float_as_uint(v);
    if (v != v) b = 0xFF800000u;
    if ((b << 1) == 0u) b = 0u;
    const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    return ((unsigned long long)ord << 32) | (unsigned long long)(0xFFFFFFFFu - n);
}

// Whole-warp maximum of the lanes' keys, folded into *dst by one lane.
__device__ __forceinline__ void argmax_warp(unsigned long long *dst, unsigned long long key) {
#pragma unroll
    for (int off = 16; off; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, off);
        key = o > key ? o : key;
    }
    if ((threadIdx.x & 31u) == 0u && key != 0ull) atomicMax(dst, key);
}

}  // namespace dev
}  // namespace w12
