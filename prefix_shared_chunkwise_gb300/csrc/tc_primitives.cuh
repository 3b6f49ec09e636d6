// sm_103a building blocks written as inline PTX: tensor memory (TMEM) allocation,
// tcgen05.mma (bf16 operands from shared memory, fp32 accumulators in TMEM),
// completion tracking through mbarriers (every wait bounded), and TMEM <-> register
// moves.  Operand tiles live in shared memory in the 128-byte-swizzled K-major layout:
// rows of 64 bf16 (128 B) per "atom column", 8-row groups 1024 B apart, the 16-byte
// chunk j of row r stored at chunk position j ^ (r % 8).
#pragma once
#include <cuda_bf16.h>
#include <cstdint>

namespace harts {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- shared-memory operand layout -----------------------------------------------------

// Byte offset of element (row, col) in a K-major SW128 tile of `rows` rows whose K
// extent is split into atoms of 64 columns (each atom: rows x 128 B, 1024-B aligned).
__device__ __forceinline__ uint32_t sw128_offset(int rows, int row, int col) {
    const int atom = col >> 6, c = col & 63;
    return static_cast<uint32_t>(atom * rows * 128 + row * 128 +
                                 ((((c >> 3) ^ (row & 7)) << 4) | ((c & 7) << 1)));
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);          // start address
    d |= static_cast<uint64_t>(1) << 16;                         // leading offset (unused)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                 // stride offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                         // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                         // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator.  a_mn / b_mn
// select the MN-major (transposed) reading of the operand.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false,
                                                  bool b_mn = false) {
    return (1u << 4)                                   // D format: f32
         | (1u << 7)                                   // A format: bf16
         | (1u << 10)                                  // B format: bf16
         | (a_mn ? (1u << 15) : 0u)
         | (b_mn ? (1u << 16) : 0u)
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Descriptor for reading a SW128 tile stored as [K rows][MN columns] (a K-major tile
// of another product, read transposed): 64-column atoms `atom_bytes` apart, 8-row
// groups 1024 B apart.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t atom_bytes) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);
    d |= static_cast<uint64_t>((atom_bytes >> 4) & 0x3FFF) << 16;   // next 64 MN columns
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                    // next 8 K rows
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Operand of a tile product: base address, atom stride, and whether it is read MN-major
// (stored [K][MN]) or K-major (stored [MN][K]).
struct Opnd {
    uint32_t saddr, atom_bytes;
    bool mn;
};

__device__ __forceinline__ uint64_t opnd_desc(const Opnd &o, int kk) {
    // K-major: 16 K-columns = 32 B inside an atom, atoms every 4 steps.
    // MN-major: 16 K-rows = 2048 B.
    return o.mn ? desc_sw128_mn(o.saddr + kk * 2048, o.atom_bytes)
                : desc_sw128(o.saddr + (kk >> 2) * o.atom_bytes + (kk & 3) * 32);
}

// ---- TMEM allocation (one full warp executes these) ------------------------------------

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_addr(dst_smem)), "r"(ncols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}

// ---- MMA issue (one thread) -------------------------------------------------------------

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D (+)= A B with A in TMEM (bf16 pairs: one row of A per lane, 8 columns per 16 K) and B
// from shared memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// D[M x N] (+)= A[M x K] * B[N x K]^T with both operands K-major SW128 tiles; K is a
// multiple of 16, atoms of 64 columns placed `a_atom_bytes` / `b_atom_bytes` apart.
__device__ __forceinline__ void mma_tile(uint32_t d_tmem, uint32_t a_saddr, uint32_t a_atom_bytes,
                                         uint32_t b_saddr, uint32_t b_atom_bytes, int K,
                                         uint32_t idesc, bool accumulate) {
    for (int kk = 0; kk < K / 16; ++kk) {
        const uint32_t aoff = (kk >> 2) * a_atom_bytes + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * b_atom_bytes + (kk & 3) * 32;
        mma_bf16(d_tmem, desc_sw128(a_saddr + aoff), desc_sw128(b_saddr + boff), idesc,
                 (accumulate || kk > 0) ? 1u : 0u);
    }
}

// D[M x N] (+)= op(A) * op(B)^T for any mix of K-major / MN-major operands.
__device__ __forceinline__ void mma_op(uint32_t d_tmem, const Opnd &a, const Opnd &b, int M, int N,
                                       int K, bool accumulate) {
    const uint32_t id = idesc_bf16(M, N, a.mn, b.mn);
    for (int kk = 0; kk < K / 16; ++kk)
        mma_bf16(d_tmem, opnd_desc(a, kk), opnd_desc(b, kk), id, (accumulate || kk > 0) ? 1u : 0u);
}

// Arrive on `bar` when every tcgen05 operation issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Make this thread's ordinary shared-memory writes visible to the tensor cores.
__device__ __forceinline__ void fence_smem_to_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- mbarriers --------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t phase) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(phase) : "memory");
    return ok != 0;
}

// Wait for the given phase; gives up after ~`max_cycles` SM cycles and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase,
                                          long long max_cycles = 4000000000LL) {
    if (mbar_try(bar, phase)) return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, phase)) {
        if (clock64() - t0 > max_cycles) return false;
    }
    return true;
}

// Arrive on a barrier (count 1) and add `bytes` to the transactions its phase waits for.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// Make barrier initialisation visible to the asynchronous proxy (TMA completions).
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// ---- TMA tiled loads (tensor map in kernel parameter space; completion on an mbarrier) --
// The destination must be 1024-byte aligned for the 128-byte swizzle used here; every
// coordinate passed by this library lies inside the tensor.

__device__ __forceinline__ void tma_load_2d(void *dst, const void *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const void *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(smem_addr(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z),
           "r"(smem_addr(bar))
        : "memory");
}

// ---- TMA tiled stores (completion tracked by bulk async-groups of the issuing thread) ----
// The source tile is 1024-byte aligned and laid out as the map's box (128-byte swizzle);
// the threads that wrote it fence it to the async proxy and meet before one thread issues
// the store.  Every coordinate passed by this library lies inside the tensor.

__device__ __forceinline__ void tma_store_2d(const void *map, int x, int y, const void *src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];"
                 :: "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(src)) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's committed stores have been read (reusable)
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's committed stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- TMEM <-> registers (warp-collective; warp w may touch lanes 32*(w%4)..+31) ---------

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t *u = reinterpret_cast<uint32_t *>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]),
          "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]),
          "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]),
          "=r"(u[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    uint32_t *u = reinterpret_cast<uint32_t *>(r);
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]),
          "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]),
          "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Two 32-column TMEM loads of one warp, issued back to back and waited for once; the wait
// names the destination registers so that no use of them can move above it.
__device__ __forceinline__ void tmem_ld32_issue(uint32_t taddr, uint32_t (&u)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]), "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]), "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]), "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld32x2(uint32_t (&a)[32], uint32_t (&b)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]), "+r"(a[6]), "+r"(a[7]), "+r"(a[8]), "+r"(a[9]), "+r"(a[10]), "+r"(a[11]), "+r"(a[12]), "+r"(a[13]), "+r"(a[14]), "+r"(a[15]), "+r"(a[16]), "+r"(a[17]), "+r"(a[18]), "+r"(a[19]), "+r"(a[20]), "+r"(a[21]), "+r"(a[22]), "+r"(a[23]), "+r"(a[24]), "+r"(a[25]), "+r"(a[26]), "+r"(a[27]), "+r"(a[28]), "+r"(a[29]), "+r"(a[30]), "+r"(a[31]),
                   "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]), "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7]), "+r"(b[8]), "+r"(b[9]), "+r"(b[10]), "+r"(b[11]), "+r"(b[12]), "+r"(b[13]), "+r"(b[14]), "+r"(b[15]), "+r"(b[16]), "+r"(b[17]), "+r"(b[18]), "+r"(b[19]), "+r"(b[20]), "+r"(b[21]), "+r"(b[22]), "+r"(b[23]), "+r"(b[24]), "+r"(b[25]), "+r"(b[26]), "+r"(b[27]), "+r"(b[28]), "+r"(b[29]), "+r"(b[30]), "+r"(b[31])
                 :: "memory");
}

__device__ __forceinline__ void tmem_ld32x2(uint32_t ta, float (&ra)[32], uint32_t tb, float (&rb)[32]) {
    uint32_t(&ua)[32] = reinterpret_cast<uint32_t(&)[32]>(ra);
    uint32_t(&ub)[32] = reinterpret_cast<uint32_t(&)[32]>(rb);
    tmem_ld32_issue(ta, ua);
    tmem_ld32_issue(tb, ub);
    tmem_wait_ld32x2(ua, ub);
}

// 32 columns of one TMEM lane per thread, without waiting for the store.
__device__ __forceinline__ void tmem_st32_issue(uint32_t taddr, const float (&r)[32]) {
    const uint32_t *u = reinterpret_cast<const uint32_t *>(r);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]), "r"(u[6]), "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]), "r"(u[13]), "r"(u[14]), "r"(u[15]), "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]), "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]), "r"(u[24]), "r"(u[25]), "r"(u[26]), "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31])
        : "memory");
}

// Two 32-column TMEM stores of one warp, then one wait.
__device__ __forceinline__ void tmem_st32x2(uint32_t ta, const float (&ra)[32], uint32_t tb, const float (&rb)[32]) {
    tmem_st32_issue(ta, ra);
    tmem_st32_issue(tb, rb);
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&r)[32]) {
    const uint32_t *u = reinterpret_cast<const uint32_t *>(r);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(u[0]), "r"(u[1]), "r"(u[2]), "r"(u[3]), "r"(u[4]), "r"(u[5]),
           "r"(u[6]), "r"(u[7]), "r"(u[8]), "r"(u[9]), "r"(u[10]), "r"(u[11]), "r"(u[12]),
           "r"(u[13]), "r"(u[14]), "r"(u[15]), "r"(u[16]), "r"(u[17]), "r"(u[18]), "r"(u[19]),
           "r"(u[20]), "r"(u[21]), "r"(u[22]), "r"(u[23]), "r"(u[24]), "r"(u[25]), "r"(u[26]),
           "r"(u[27]), "r"(u[28]), "r"(u[29]), "r"(u[30]), "r"(u[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Pack two floats to a bf16x2 word (lower address = first).
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// Store 8 consecutive K-columns (col % 8 == 0) of one row into a SW128 tile (16 B).
__device__ __forceinline__ void st_sw128_8(uint8_t *tile, int rows, int row, int col,
                                           const float *v) {
    uint4 w;
    w.x = pack_bf16(v[0], v[1]); w.y = pack_bf16(v[2], v[3]);
    w.z = pack_bf16(v[4], v[5]); w.w = pack_bf16(v[6], v[7]);
    *reinterpret_cast<uint4 *>(tile + sw128_offset(rows, row, col)) = w;
}

}  // namespace tc
}  // namespace harts

namespace harts {
namespace tc {

// ---- asynchronous global -> shared copies (16 B; zero-filled when src_bytes == 0) -------

__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;"
                 :: "r"(smem_addr(dst_smem)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst_smem, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;"
                 :: "r"(smem_addr(dst_smem)), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

}  // namespace tc
}  // namespace harts
