// Token-batch FFN on the tensor cores (tcgen05, TMEM), the S-MoE page "Metal
// Compute Kernels", section "Token-Batch Fused FFN": for T tokens the three
// projections are dense contractions, Y = W X^T with the weights' K axis
// contracted against every token.  One launch set serves the token batches
// of up to 32 experts (the page's batch per claimed expert): their token
// tiles are concatenated along the grid's y axis.
//
// Exactness plan (the scale varies per (row, group), so it cannot be folded
// into an operand):
//  * A (weights, 128 rows x 64 columns per K tile, one group slice) holds
//    each code c as the exact bf16 value (c - Z)/DEN: Q4 (c - 7.5)/16 =
//    (2c - 15)/32 (an odd numerator of at most 4 bits), made from the exact
//    bf16 1 + c/16 (a bit pattern) minus 1.46875; Q2 (c - 1.5)/4 from
//    1 + c/4 minus 1.375.  Each subtraction's exact result is representable.
//    Per 64-column tile of one group the accumulator is then
//    D = sum (c - Z) x / DEN and sum w x = s sum (c - Z) x / Z = s (DEN/Z) D.
//  * B (tokens, NT x 64) holds x split into two bf16 halves, hi = bf16(x) and
//    lo = bf16(x - hi), stored as one operand of 2 NT rows (hi rows, then
//    lo rows), x represented to about 2^-17 relative.  Token tiles of 128:
//    per K step one MMA of N = 128 takes the hi rows and a second the lo
//    rows, accumulating into the same 128 columns, so an accumulator takes
//    128 TMEM columns.  Smaller tiles: one MMA of N = 2 NT computes both halves into
//    2 NT columns and the epilogue adds the hi and lo columns (two MMAs of a
//    small N cost more than one of twice the N).
//  * Each 64-column tile's accumulator is read back from TMEM and added to
//    per-thread f32 sums with the tile's scale.  TMEM holds several tiles'
//    accumulators, so the MMAs run ahead of the epilogue.
//  * A goes straight into TMEM (tcgen05.st; up to 8 stages after 256
//    columns of accumulators, or 4 after 128 when two CTAs share an SM) and
//    the MMAs read it there, which leaves shared memory to the token blocks
//    (the canonical no-swizzle K-major layout).
//
// Three launches per call, chained with programmatic dependent launch:
//  1. prep_tokens: X -> B blocks (hi, lo per (token tile, K tile)).
//  2. tc_ffn<BITS, NT, gate/up>: a CTA tile is 64 gate rows + the same 64 up
//     rows (128 accumulator rows) over one K range.  The K splits of a tile
//     form one thread-block cluster: each split leaves its partial sums in
//     its shared memory, then split q adds token columns [q NT/S, (q+1)
//     NT/S) of every split's partials (in split order, read through
//     distributed shared memory), forms SiLU(g) * u and writes it directly
//     as the B block of the down projection's K tile (64 hidden columns =
//     one down K tile).  Its code-streaming warp also prefetches the down
//     weights into L2 once its own chunks are out.
//  3. tc_ffn<BITS, NT, down>: 128 down rows over one K range, split the same
//     way; each split writes Y for its token columns.
// Inside a GEMM CTA (640 threads): warps 0-7 epilogue (warp w reads TMEM
// lane quarter w % 4 = 32 tile rows, columns of half w / 4), warps 8-15
// convert codes to A tiles in two groups of four that take alternate K
// tiles (thread = one tile row), warps 16 and 19 issue the MMAs of even and
// odd K tiles, warp 17 streams code chunks with 2-D tensor copies (TMA,
// 128-byte swizzle: 128 bytes x 64 or 128 rows per chunk), warp 18 streams
// the token B blocks with bulk copies.
// Two converter and two epilogue warps per SM sub-partition keep those
// dependent chains overlapped.  Every hand-off is an mbarrier with one
// in-order waiter per role, so each awaited phase parity is unambiguous;
// every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"
#include "internal.h"

namespace smoe {
namespace {

constexpr int KT = 64;                        // columns per K tile (one group slice)
constexpr int MT = 128;                       // accumulator rows per CTA tile
// K tiles per code chunk: a chunk row is 128 bytes of codes (Q4: 4 tiles
// of 64 columns, Q2: 8).
template <int BITS>
constexpr int chunk_kt() { return 128 / (KT * BITS / 8); }
constexpr uint32_t CHUNK_BYTES = MT * 128u;   // 128 rows x 128 bytes of Q4 codes
constexpr int CODE_SLOTS = 3;
constexpr int EPI_WARPS = 8;
constexpr int CONV_WARPS = 8;
constexpr int CONV_WARP0 = 8;
constexpr int MMA_WARP = 16;    // issues the MMAs of even K tiles (and owns the TMEM allocation)
constexpr int CODE_WARP = 17;
constexpr int BPROD_WARP = 18;
constexpr int MMA_WARP2 = 19;   // issues the MMAs of odd K tiles
constexpr int TC_THREADS = 20 * 32;
// A holds (c - Z) / DEN exactly (DEN = 16 at Q4, 4 at Q2), so per group
// sum w x = s (DEN / Z) sum A x: FOLD = DEN / Z.
template <int BITS>
constexpr float fold() { return BITS == 4 ? 16.0f / 7.5f : 4.0f / 1.5f; }
constexpr int TC_MAX_EXPERTS = 32;  // experts per launch (grouped token batch)

// B block of one (token tile, K tile): hi [NT x 64] bf16, then lo.
__host__ __device__ constexpr uint32_t b_bytes(int nt) { return static_cast<uint32_t>(nt) * 256u; }
__host__ __device__ constexpr uint32_t round1024(uint32_t v) { return (v + 1023u) & ~1023u; }
// hi and lo accumulated into the same columns (token tiles of 128)
__host__ __device__ constexpr bool hilo_shared(int nt) { return nt == 128; }
// TMEM columns of one accumulator
__host__ __device__ constexpr int acc_cols(int nt) { return hilo_shared(nt) ? nt : 2 * nt; }
// The converters store A straight into tensor memory (stages of 32 columns
// after the accumulators), so a K tile's A makes no round trip through
// shared memory and the MMAs read only the token block there (measured
// against A in shared memory: 2% faster at T = 256 and 3% at T = 64, once
// the converters no longer paced the loop).  A CTA takes all 512 columns
// (256 of accumulators, up to 8 A stages) and holds an SM alone; with tiles
// of 16 and more tiles than SMs, a CTA takes 256 (128 of accumulators, 4 A
// stages) so that two share an SM (`two`): two CTAs per SM give each a
// slower K loop, so this pays only where the tiles would otherwise run in
// more waves.
__host__ __device__ constexpr uint32_t a_tmem_col0(bool two) { return two ? 128u : 256u; }
// Stage and accumulator-buffer counts are even: K tiles i and i + S (or
// i + NB) then always belong to the same MMA issuer and converter group, so
// every barrier phase has one in-order waiter.
__host__ __device__ constexpr int tc_accbufs(int nt, bool two)
{
    return static_cast<int>(a_tmem_col0(two)) / acc_cols(nt) < 8 ? static_cast<int>(a_tmem_col0(two)) / acc_cols(nt)
                                                                   : 8;
}
// A stage in shared memory holds one token block.
__host__ __device__ constexpr uint32_t tc_stage_bytes(int nt) { return round1024(b_bytes(nt)); }
constexpr size_t kTcSmemBudget = 224 * 1024;
__host__ __device__ constexpr int tc_stages(int nt, bool two)
{
    return two ? 4
               : ((kTcSmemBudget - CODE_SLOTS * CHUNK_BYTES - 2048) / tc_stage_bytes(nt) < 8
                      ? static_cast<int>((kTcSmemBudget - CODE_SLOTS * CHUNK_BYTES - 2048) / tc_stage_bytes(nt))
                      : 8) & ~1;
}

// Byte offset of (row, 8-column block k8) in a [rows x 64] bf16 tile laid out
// as 8x8 core matrices: core (row/8, k8) at ((row/8)*8 + k8)*128, row%8 at 16*(row%8).
__host__ __device__ __forceinline__ uint32_t core_off(int row, int k8)
{
    return static_cast<uint32_t>(((row >> 3) * 8 + k8) * 128 + (row & 7) * 16);
}

// The K order inside a tile follows the order in which a 32-bit code word
// unpacks to bf16 pairs; B uses the same order, so the contraction is
// unchanged.  Column of position p (0..7) of 8-column block kb of a tile:
//  Q4: a word is 8 columns, one block, order 0,4,1,5,2,6,3,7;
//  Q2: a word is 16 columns, two blocks, pairs (i, i + 8): block 2w holds
//      0,8,1,9,2,10,3,11 of word w and block 2w + 1 holds 4,12,...,7,15.
__host__ __device__ __forceinline__ int tile_col(int bits, int kb, int p)
{
    if (bits == 4) return 8 * kb + ((p & 1) ? 4 + (p >> 1) : (p >> 1));
    return 16 * (kb >> 1) + 4 * (kb & 1) + (p >> 1) + 8 * (p & 1);
}

// tcgen05 shared-memory matrix descriptor, no swizzle, K-major:
// LBO = distance between core matrices along K (128 B), SBO = between 8-row
// groups (1024 B), version field 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr)
{
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(128u >> 4) << 16) |
           (static_cast<uint64_t>(1024u >> 4) << 32) | (static_cast<uint64_t>(1) << 46);
}

// Instruction descriptor, kind::f16: f32 accumulate, A and B bf16, both
// K-major, N at bit 17 (in 8s), M at bit 24 (in 16s).
__host__ __device__ constexpr uint32_t instr_desc(int m, int n)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

// tcgen05 MMA, kind::f16, A read from tensor memory (M = 128 rows in the
// 128 lanes, K along the columns, two bf16 per 32-bit column), B from a
// shared-memory descriptor, D in tensor memory.
__device__ __forceinline__ void mma_bf16_ta(uint32_t tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 TMEM lanes (this
// thread's lane), from registers.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::
            "r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void mma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 8 consecutive f32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v)
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive f32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v)
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// N (a multiple of 8) consecutive f32 columns of this warp's 32 TMEM lanes.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float (&v)[N])
{
#pragma unroll
    for (int c = 0; c + 32 <= N; c += 32) tmem_ld32(taddr + c, v + c);
#pragma unroll
    for (int c = N / 32 * 32; c < N; c += 8) tmem_ld8(taddr + c, v + c);
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// bf16x2 a - b (round to nearest; exact here: the difference is representable).
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// One 32-bit word of Q4 codes (columns 0..7) as 8 exact bf16 values
// (c - 7.5)/16, in the order 0,4,1,5,2,6,3,7: the bit pattern of 1 + c/16
// (exponent 0, c in the top four mantissa bits) minus 1 + 7.5/16.
__device__ __forceinline__ uint4 q4_word_to_bf16(uint32_t w)
{
    const uint32_t mag = 0x3F803F80u;  // 1.0, 1.0
    const uint32_t off = 0x3FBC3FBCu;  // 1.46875, 1.46875
    uint4 r;
    r.x = bf16x2_sub(((w << 3) & 0x00780078u) | mag, off);  // columns 0 and 4
    r.y = bf16x2_sub(((w >> 1) & 0x00780078u) | mag, off);  // 1 and 5
    r.z = bf16x2_sub(((w >> 5) & 0x00780078u) | mag, off);  // 2 and 6
    r.w = bf16x2_sub(((w >> 9) & 0x00780078u) | mag, off);  // 3 and 7
    return r;
}

// One 32-bit word of Q2 codes (columns 0..15) as 16 exact bf16 values
// (c - 1.5)/4 in pairs (i, i + 8): the bit pattern of 1 + c/4 (c in the top
// two mantissa bits) minus 1 + 1.5/4 = 1.375.  lo: pairs 0..3, hi: 4..7.
__device__ __forceinline__ void q2_word_to_bf16(uint32_t w, uint4 &lo, uint4 &hi)
{
    const uint32_t mag = 0x3F803F80u;  // 1.0, 1.0
    const uint32_t off = 0x3FB03FB0u;  // 1.375, 1.375
    lo.x = bf16x2_sub(((w << 5) & 0x00600060u) | mag, off);  // columns 0 and 8
    lo.y = bf16x2_sub(((w << 3) & 0x00600060u) | mag, off);  // 1 and 9
    lo.z = bf16x2_sub(((w << 1) & 0x00600060u) | mag, off);  // 2 and 10
    lo.w = bf16x2_sub(((w >> 1) & 0x00600060u) | mag, off);  // 3 and 11
    hi.x = bf16x2_sub(((w >> 3) & 0x00600060u) | mag, off);  // 4 and 12
    hi.y = bf16x2_sub(((w >> 5) & 0x00600060u) | mag, off);  // 5 and 13
    hi.z = bf16x2_sub(((w >> 7) & 0x00600060u) | mag, off);  // 6 and 14
    hi.w = bf16x2_sub(((w >> 9) & 0x00600060u) | mag, off);  // 7 and 15
}

__device__ __forceinline__ uint4 lds128v(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint2 lds64v(uint32_t addr)
{
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

// L2 prefetch of one box of a 2-D tensor map at (x bytes, y rows); parts
// outside the tensor are skipped.  x must be a multiple of 16.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y)
{
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y)
                 : "memory");
}

// L2 prefetch of `bytes` (a multiple of 16) from a 16-byte aligned global address.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tensor copy global -> shared of one box at (x bytes, y rows),
// completing on the mbarrier.  x must be a multiple of 16.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Splits 8 values into bf16 hi/lo (hi = bf16(v), lo = bf16(v - hi)) packed
// in pairs.
__device__ __forceinline__ void split8(const float (&v)[8], uint32_t (&hi)[4], uint32_t (&lo)[4])
{
#pragma unroll
    for (int p = 0; p < 8; p += 2) {
        const __nv_bfloat16 h0 = __float2bfloat16_rn(v[p]);
        const __nv_bfloat16 h1 = __float2bfloat16_rn(v[p + 1]);
        const __nv_bfloat16 l0 = __float2bfloat16_rn(v[p] - __bfloat162float(h0));
        const __nv_bfloat16 l1 = __float2bfloat16_rn(v[p + 1] - __bfloat162float(h1));
        hi[p / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(h0)) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(h1)) << 16);
        lo[p / 2] = static_cast<uint32_t>(__bfloat16_as_ushort(l0)) |
                    (static_cast<uint32_t>(__bfloat16_as_ushort(l1)) << 16);
    }
}

// SiLU with the fast exponential and division intrinsics (relative error a
// few units in the last place for |v| < 100, far inside the tolerance; 0
// once exp(-v) overflows).
__device__ __forceinline__ float silu_fast(float v) { return __fdividef(v, 1.0f + __expf(-v)); }

// ---- thread-block cluster helpers (the K splits of a tile form a cluster)

// All threads of all CTAs of the cluster: arrive (release) and wait
// (acquire).  Every thread of the kernel executes each call exactly once.
__device__ __forceinline__ void cluster_sync()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The two halves of cluster_sync, for work that may run between them.
__device__ __forceinline__ void cluster_arrive()
{
    __syncwarp();
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait()
{
    __syncwarp();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The address of shared-memory location `addr` (this CTA's window) in the
// shared memory of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, int rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f32x4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// The expert owning global token tile g: the last e with tile0[e] <= g.
__device__ __forceinline__ int expert_of_tile(const int *tile0, int n, int g)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile0[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ---------------------------------------------------------------- token prep

struct PrepArgs {
    const float *X[TC_MAX_EXPERTS];   // expert e's tokens [T[e] x K]
    int T[TC_MAX_EXPERTS];
    int tile0[TC_MAX_EXPERTS + 1];    // first global token tile of each expert
    int n;                            // experts
    int bits;        // code width of the weights B is contracted with (K order)
    uint8_t *Bblk;   // [ntiles][K/64] blocks of b_bytes(nt), global token tiles
    int K, nt, ntiles;
};

// One thread per (token slot of a global tile, 8-column block): the token's 8
// values split into bf16 hi/lo in the tile layout.  Slots past an expert's T
// (padding of its last tile) are zeros.
__global__ void __launch_bounds__(256) prep_tokens(const __grid_constant__ PrepArgs a)
{
    // the next kernel may start its weight-only prologue now: everything it
    // reads from this grid it reads after its own griddepcontrol.wait
    pdl_launch_dependents();
    pdl_wait();
    const int kb_per_t = a.K / 8;
    const int nkt = a.K / KT;
    const long long total = static_cast<long long>(a.ntiles) * a.nt * kb_per_t;  // multiple of 8
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long first = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rounds = (total + stride - 1) / stride;
    for (long long rd = 0; rd < rounds; ++rd) {
        const long long idx = rd * stride + first;
        if (idx >= total) break;
        const int slot = static_cast<int>(idx / kb_per_t);  // global token slot
        const int kb = static_cast<int>(idx % kb_per_t);
        const int kt = kb / 8;
        const int k8 = kb % 8;
        const int gt = slot / a.nt;
        const int e = expert_of_tile(a.tile0, a.n, gt);
        const int t = (gt - a.tile0[e]) * a.nt + slot % a.nt;  // the expert's token
        float v[8];
        if (t < a.T[e]) {
            const float *src = a.X[e] + static_cast<size_t>(t) * a.K + static_cast<size_t>(kt) * KT;
            if (a.bits == 4) {
                // the block's 8 contiguous columns, permuted in registers
                const float4 *q = reinterpret_cast<const float4 *>(src + 8 * k8);
                const float4 p0 = q[0], p1 = q[1];
                const float raw[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
                for (int p = 0; p < 8; ++p) v[p] = raw[tile_col(4, k8, p) - 8 * k8];
            } else {
                // 8 of the 16 columns of the block's code word
                const float4 *q = reinterpret_cast<const float4 *>(src + 16 * (k8 >> 1));
                const float4 p0 = q[0], p1 = q[1], p2 = q[2], p3 = q[3];
                const float raw[16] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w,
                                       p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
#pragma unroll
                for (int p = 0; p < 8; ++p) v[p] = raw[tile_col(2, k8, p) - 16 * (k8 >> 1)];
            }
        } else {
#pragma unroll
            for (int p = 0; p < 8; ++p) v[p] = 0.f;
        }
        uint32_t hi[4], lo[4];
        split8(v, hi, lo);
        uint8_t *blk = a.Bblk + (static_cast<size_t>(gt) * nkt + kt) * b_bytes(a.nt);
        const uint32_t off = core_off(slot % a.nt, k8);
        *reinterpret_cast<uint4 *>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(blk + static_cast<size_t>(a.nt) * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// ---------------------------------------------------------------- GEMM

// One GEMM launch over the token tiles of n experts: global token tile g
// belongs to the expert e with tile0[e] <= g < tile0[e + 1].
struct alignas(128) TcArgs {  // CUtensorMap members are 128-byte aligned
    CUtensorMap tmap[TC_MAX_EXPERTS][2];  // codes: gate and up rows (gate/up) or down rows ([e][0])
    const float *scales[TC_MAX_EXPERTS][2];
    float *Y[TC_MAX_EXPERTS];             // down: [T[e] x M]
    int T[TC_MAX_EXPERTS];
    int tile0[TC_MAX_EXPERTS + 1];
    const uint8_t *B;       // token operand blocks [ntiles][K/64] (global tiles)
    uint8_t *Hb;            // gate/up: down-operand blocks [ntiles][M/64]
    unsigned *status;
    int n;                  // experts
    int M;                  // rows per matrix (d_ff for gate/up, d_model for down)
    int K, group, ntiles, kps, nsplit;
    // gate/up: the down projection's codes (boxes of 128 rows x 128 bytes)
    // and scales, which the CTAs prefetch into L2 for the next launch
    CUtensorMap pmap[TC_MAX_EXPERTS];
    const float *pscales[TC_MAX_EXPERTS];  // null: not prefetched
    int pM, pK;                            // down rows (d_model) and columns (d_ff); pK = 0: no prefetch
};
static_assert(sizeof(TcArgs) <= 32764, "kernel parameters are limited to 32,764 bytes");

// Gate/up finish: the hidden values of tokens [n0, n1) of this tile (global
// token tile gtile, the expert's tile ltile of an expert with Te tokens),
// src[(n - n0) stride + c] for hidden column c (0..63), written as the bf16
// hi/lo B block of down K tile `mtile` (tokens past Te as zeros).  Work item: (token,
// 8-column block), spread over threads et = 0 .. nthreads - 1.
template <int BITS, int NT>
__device__ __forceinline__ void write_hidden_block(const TcArgs &a, const float *src, int stride, int mtile,
                                                   int gtile, int ltile, int Te, int n0, int n1, int et,
                                                   int nthreads)
{
    uint8_t *blk = a.Hb + (static_cast<size_t>(gtile) * (a.M / KT) + mtile) * b_bytes(NT);
    for (int it = et; it < (n1 - n0) * 8; it += nthreads) {
        const int n = n0 + (it >> 3), k8 = it & 7;
        const int t = ltile * NT + n;
        float v[8];
#pragma unroll
        for (int p = 0; p < 8; ++p) v[p] = t < Te ? src[(n - n0) * stride + tile_col(BITS, k8, p)] : 0.f;
        uint32_t hi[4], lo[4];
        split8(v, hi, lo);
        const uint32_t off = core_off(n, k8);
        *reinterpret_cast<uint4 *>(blk + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(blk + static_cast<size_t>(NT) * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

template <int BITS, int NT, bool GU, bool TWO>
__global__ void __launch_bounds__(TC_THREADS, TWO ? 2 : 1) tc_ffn(const __grid_constant__ TcArgs a)
{
    constexpr int CHUNK_KT = chunk_kt<BITS>();
    constexpr int TILE_BYTES = KT * BITS / 8;  // bytes of one row's codes per K tile
    static_assert(!TWO || NT == 16, "two CTAs per SM only with 16-token tiles");
    static_assert(tc_stages(NT, TWO) % 2 == 0 && tc_accbufs(NT, TWO) % 2 == 0,
                  "even stage and buffer counts: one waiter per barrier phase with two MMA issuers");
    constexpr int NB = tc_accbufs(NT, TWO);
    constexpr uint32_t ACOL0 = a_tmem_col0(TWO);  // first A stage column
    constexpr bool HL = hilo_shared(NT);
    constexpr int AC = acc_cols(NT);  // TMEM columns of one accumulator
    constexpr uint32_t NCOLS = 2u * ACOL0;  // accumulators, then the A stages
    constexpr int S = tc_stages(NT, TWO);
    constexpr uint32_t SB = tc_stage_bytes(NT);
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t codes0 = base;                              // CODE_SLOTS chunks, 1024-aligned
    const uint32_t stage0 = base + CODE_SLOTS * CHUNK_BYTES;   // S stages of A + B
    const uint32_t bars = stage0 + S * SB;
    const uint32_t cfull0 = bars, cempty0 = cfull0 + 8 * CODE_SLOTS, full0 = cempty0 + 8 * CODE_SLOTS,
                   empty0 = full0 + 8 * S, accf0 = empty0 + 8 * S, acce0 = accf0 + 8 * NB, tslot = acce0 + 8 * NB;
    uint32_t *tmem_word = reinterpret_cast<uint32_t *>(smem_raw + (tslot - raw));

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int mtile = blockIdx.x;
    const int gtile = blockIdx.y;  // global token tile
    const int xe = expert_of_tile(a.tile0, a.n, gtile);
    const int ltile = gtile - a.tile0[xe];  // the expert's token tile
    const int Te = a.T[xe];
    const int split = blockIdx.z;
    const int nkt = a.K / KT;
    const int kt0 = split * a.kps;
    const int kt1 = min(nkt, kt0 + a.kps);
    const int nk = kt1 > kt0 ? kt1 - kt0 : 0;
    const int nchunks = (nk + CHUNK_KT - 1) / CHUNK_KT;
    const int ngroups = a.K / a.group;
    // code chunk c into its slot (the weights never depend on an earlier kernel)
    auto issue_chunk = [&](int c) {
        const int slot = c % CODE_SLOTS;
        const uint32_t dst = codes0 + slot * CHUNK_BYTES;
        const int x = (kt0 + c * CHUNK_KT) * TILE_BYTES;  // byte offset along the row: multiple of 16
        mbar_arrive_expect_tx(cfull0 + 8 * slot, CHUNK_BYTES);
        if (GU) {
            tma_load_2d(dst, &a.tmap[xe][0], x, mtile * 64, cfull0 + 8 * slot);
            tma_load_2d(dst + CHUNK_BYTES / 2, &a.tmap[xe][1], x, mtile * 64, cfull0 + 8 * slot);
        } else {
            tma_load_2d(dst, &a.tmap[xe][0], x, mtile * MT, cfull0 + 8 * slot);
        }
    };
    // the first CODE_SLOTS chunks go out as soon as their barriers exist,
    // before the tensor-memory allocation and the block barrier (about half
    // a microsecond earlier; the first chunk's DRAM latency is on every
    // call's critical path)
    const int early_chunks = nchunks < CODE_SLOTS ? nchunks : CODE_SLOTS;

    if (threadIdx.x == 0) {
        for (int c = 0; c < CODE_SLOTS; ++c) {
            mbar_init(cfull0 + 8 * c, 1);
            mbar_init(cempty0 + 8 * c, CONV_WARPS);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(full0 + 8 * s, CONV_WARPS / 2 + 1);  // one converter group + the token block
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < NB; ++b) {
            mbar_init(accf0 + 8 * b, 1);
            mbar_init(acce0 + 8 * b, EPI_WARPS);
        }
        fence_mbar_init();
        for (int c = 0; c < early_chunks; ++c) issue_chunk(c);
    }
    if (warp == MMA_WARP) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(tslot), "r"(NCOLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_word;
    // A wait that gives up ends its role's loop and sets `failed`; `issued`
    // counts the copies (code chunks, token blocks) or MMA groups the role
    // started, so that they can be waited for before the CTA releases its
    // shared and tensor memory.
    bool failed = false;
    int issued = 0;
    // Gate/up lets the down projection start its weight-only prologue now (it
    // lands on SMs this grid does not hold: one CTA fills an SM); whatever it
    // reads from this grid, and whatever it overwrites that this grid reads,
    // it touches only after its own griddepcontrol.wait.  The down projection
    // triggers at its end: a following call's token prep started early only
    // competed with it (measured).
    if (GU && threadIdx.x == 0) pdl_launch_dependents();

    if (warp == CODE_WARP) {
        // ---- code chunks (weights never depend on an earlier kernel)
        if (lane == 0) {
            issued = early_chunks;  // issued by thread 0 with the barriers
            for (int c = early_chunks; c < nchunks; ++c, ++issued) {
                const int slot = c % CODE_SLOTS;
                if (!mbar_wait_bounded(cempty0 + 8 * slot, ((c / CODE_SLOTS) - 1) & 1, a.status, 7u)) {
                    failed = true;
                    break;
                }
                issue_chunk(c);
            }
            if (GU && !failed && ltile == 0 && a.pK > 0) {
                // The down projection reads this expert's down weights right
                // after this launch; this one leaves DRAM mostly idle at
                // small T, so its CTAs (all issued chunks out) fetch them
                // into L2 now: each CTA a share of the 128-row x 128-byte
                // boxes and of the scales.
                const int rank = mtile + static_cast<int>(gridDim.x) * split;
                const int nr = static_cast<int>(gridDim.x * gridDim.z);
                const int rb = (a.pM + MT - 1) / MT, cb = (a.pK * BITS / 8 + 127) / 128;
                for (int bx = rank; bx < rb * cb; bx += nr) tma_prefetch_2d(&a.pmap[xe], (bx % cb) * 128, (bx / cb) * MT);
                if (a.pscales[xe]) {
                    const size_t sb = static_cast<size_t>(a.pM) * (a.pK / a.group) * sizeof(float);  // multiple of 16
                    const uint8_t *sp = reinterpret_cast<const uint8_t *>(a.pscales[xe]);
                    for (size_t off = static_cast<size_t>(rank) * 4096u; off < sb; off += static_cast<size_t>(nr) * 4096u)
                        bulk_prefetch_l2(sp + off, static_cast<uint32_t>(sb - off < 4096u ? sb - off : 4096u));
                }
            }
        }
    } else if (warp == BPROD_WARP) {
        // ---- token blocks, produced by the previous kernel
        pdl_wait();
        if (lane == 0) {
            const uint8_t *src = a.B + (static_cast<size_t>(gtile) * nkt + kt0) * b_bytes(NT);
            for (int i = 0; i < nk; ++i, ++issued) {
                const int s = i % S;
                if (i >= S && !mbar_wait_bounded(empty0 + 8 * s, ((i / S) - 1) & 1, a.status, 8u)) {
                    failed = true;
                    break;
                }
                mbar_arrive_expect_tx(full0 + 8 * s, b_bytes(NT));
                bulk_g2s(stage0 + s * SB, src + static_cast<size_t>(i) * b_bytes(NT), b_bytes(NT),
                         full0 + 8 * s);
            }
        }
    } else if (warp == MMA_WARP || warp == MMA_WARP2) {
        // ---- MMA issue: two issuing threads take alternate K tiles, so
        // one's barrier waits and commits overlap the other's MMAs (one
        // issuer spent more than half of each tile's time outside the MMAs)
        if (lane == 0) {
            const uint32_t idesc = instr_desc(MT, HL ? NT : 2 * NT);
            constexpr uint32_t LO = static_cast<uint32_t>(NT) * 128u;  // the lo rows of a token block
            const int i0 = warp == MMA_WARP ? 0 : 1;
            for (int i = i0; i < nk; i += 2, ++issued) {
                const int s = i % S, b = i % NB;
                const uint32_t spar = static_cast<uint32_t>(i / S) & 1u, bpar = static_cast<uint32_t>(i / NB) & 1u;
                if (!mbar_wait_bounded(full0 + 8 * s, spar, a.status, 3u) ||
                    (i >= NB && !mbar_wait_bounded(acce0 + 8 * b, bpar ^ 1u, a.status, 4u))) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t sb = stage0 + s * SB;  // the token block
                const uint32_t d = tmem + static_cast<uint32_t>(b * AC);
#pragma unroll
                for (int kk = 0; kk < KT / 16; ++kk) {
                    const uint32_t at = tmem + ACOL0 + static_cast<uint32_t>(s * 32 + kk * 8);
                    mma_bf16_ta(d, at, smem_desc(sb + kk * 256), idesc, kk != 0);
                    if (HL) mma_bf16_ta(d, at, smem_desc(sb + LO + kk * 256), idesc, 1u);
                }
                mma_commit(empty0 + 8 * s);
                mma_commit(accf0 + 8 * b);
            }
        }
    } else if (warp >= CONV_WARP0) {
        // ---- codes -> A tiles.  The converter warps form two groups of four
        // (each group covers the 128 tile rows, i.e. all four TMEM lane
        // quarters); group g converts the K tiles i with i % 2 == g, so two
        // tiles are in conversion at once (one group of eight warps on one
        // tile at a time paced the K loop: 0.3-0.4 us of conversion latency
        // per tile).  Thread (g, r) converts the whole tile row r.
        const int ct = threadIdx.x - CONV_WARP0 * 32;
        const int r = ct & (MT - 1), grp = ct >> 7;
        const uint32_t rsw = static_cast<uint32_t>(r & 7);  // 128-byte swizzle of the chunk rows
        for (int i = grp; i < nk; i += 2) {
            // K tile i: tile `sub` of chunk c in code slot `slot` (fill
            // parity cpar), stage s (round parity spar)
            const int c = i / CHUNK_KT, sub = i - c * CHUNK_KT;
            const int slot = c % CODE_SLOTS;
            const uint32_t cpar = static_cast<uint32_t>(c / CODE_SLOTS) & 1u;
            const int s = i % S;
            const uint32_t spar = static_cast<uint32_t>(i / S) & 1u;
            // the group's first tile of a chunk waits for the chunk (chunks
            // start at even tiles: that tile is sub == grp)
            if ((sub == grp && !mbar_wait_bounded(cfull0 + 8 * slot, cpar, a.status, 5u)) ||
                (i >= S && !mbar_wait_bounded(empty0 + 8 * s, spar ^ 1u, a.status, 5u))) {
                failed = true;
                break;
            }
            const uint32_t row = codes0 + slot * CHUNK_BYTES + static_cast<uint32_t>(r) * 128u;
            tc_fence_after();  // after the wait for the MMA that last read this stage
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                // 16 columns (32 bf16) of tile row r, in the K order of
                // the B operand, straight into tensor memory
                uint32_t v[16];
                if (BITS == 4) {
                    const uint4 w = lds128v(row + (((2u * sub + static_cast<uint32_t>(hf)) ^ rsw) << 4));
                    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint4 cv = q4_word_to_bf16(words[q]);
                        v[4 * q] = cv.x; v[4 * q + 1] = cv.y; v[4 * q + 2] = cv.z; v[4 * q + 3] = cv.w;
                    }
                } else {
                    const uint2 w = lds64v(row + ((static_cast<uint32_t>(sub) ^ rsw) << 4) + 8u * hf);
                    const uint32_t words[2] = {w.x, w.y};
#pragma unroll
                    for (int q = 0; q < 2; ++q) {
                        uint4 lo, hi;
                        q2_word_to_bf16(words[q], lo, hi);
                        v[8 * q] = lo.x; v[8 * q + 1] = lo.y; v[8 * q + 2] = lo.z; v[8 * q + 3] = lo.w;
                        v[8 * q + 4] = hi.x; v[8 * q + 5] = hi.y; v[8 * q + 6] = hi.z; v[8 * q + 7] = hi.w;
                    }
                }
                tmem_st16(tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + ACOL0 +
                              static_cast<uint32_t>(s * 32 + 16 * hf),
                          v);
            }
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(full0 + 8 * s);
                // the group's last tile of the chunk releases the code slot
                // (a group without a tile in the final chunk never arrives
                // there; nothing waits for that slot again)
                if (sub + 2 >= CHUNK_KT || i + 2 >= nk) mbar_arrive(cempty0 + 8 * slot);
            }
        }
    } else {
        // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (= tile
        // rows) and columns [h NH, (h + 1) NH) of each accumulator, h = w / 4.
        // It writes partials, hidden blocks and Y: all after the previous
        // kernel has completed.
        pdl_wait();
        constexpr int NH = NT / 2;
        const int q = warp & 3, h = warp >> 2;
        const int r = q * 32 + lane;
        const int et = h * MT + r;  // 0..255 over the epilogue threads
        const int mat = GU ? (r >> 6) : 0;
        const int row = GU ? mtile * 64 + (r & 63) : mtile * MT + r;
        const bool rok = row < a.M;
        const float *srow = a.scales[xe][mat] + static_cast<size_t>(rok ? row : 0) * ngroups;
        float y[NH];
#pragma unroll
        for (int n = 0; n < NH; ++n) y[n] = 0.f;
        // scale group gnext holds the next K tile to fold, its rnext-th of tpg
        const int tpg = a.group / KT;
        int gnext = kt0 / tpg, rnext = kt0 - gnext * tpg;
        float sc_next = (rok && nk > 0) ? ldg_f32(srow + gnext) : 0.f;
        int b = 0;
        uint32_t bpar = 0;  // accumulator buffer b, round parity
        for (int i = 0; i < nk; ++i) {
            const float f = sc_next * fold<BITS>();
            if (++rnext == tpg) {
                rnext = 0;
                ++gnext;
            }
            if (i + 1 < nk) sc_next = rok ? ldg_f32(srow + gnext) : 0.f;
            const bool ok = mbar_wait_bounded(accf0 + 8 * b, bpar, a.status, 6u);
            if (!__all_sync(FULL_MASK, ok)) {
                failed = true;
                break;
            }
            tc_fence_after();
            // columns [c, c + CH) of this warp's half, CH at a time (and,
            // when hi and lo have their own columns, the lo columns NT later)
            constexpr int CH = NH < 16 ? NH : (NH > 32 ? 8 : 16);
            const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(b * AC + h * NH);
#pragma unroll
            for (int c = 0; c < NH; c += CH) {
                float vh[CH], vl[CH];
                tmem_ld<CH>(tq + c, vh);
                if (!HL) tmem_ld<CH>(tq + NT + c, vl);
                tmem_wait_ld();
#pragma unroll
                for (int n = 0; n < CH; ++n) y[c + n] = fmaf(f, HL ? vh[n] : vh[n] + vl[n], y[c + n]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce0 + 8 * b);
            if (++b == NB) {
                b = 0;
                bpar ^= 1u;
            }
        }

        if (a.nsplit == 1) {
            // the whole K range is here: finish the tile from registers
            if (GU) {
                // rows 64..127 hold up for the hidden columns of rows 0..63:
                // exchange through shared memory (the stages are idle now),
                // then write SiLU(g) * u as the B block of down K tile `mtile`
                float *xch = reinterpret_cast<float *>(smem_raw + (stage0 - raw));  // [NT][64]
                if (r >= 64) {
#pragma unroll
                    for (int n = 0; n < NH; ++n) xch[(h * NH + n) * 64 + (r - 64)] = y[n];
                }
                named_barrier(1, EPI_WARPS * 32);
                if (r < 64) {
#pragma unroll
                    for (int n = 0; n < NH; ++n) {
                        float *p = xch + (h * NH + n) * 64 + r;
                        *p = silu_fast(y[n]) * *p;
                    }
                }
                named_barrier(1, EPI_WARPS * 32);
                write_hidden_block<BITS, NT>(a, xch, 64, mtile, gtile, ltile, Te, 0, NT, et, EPI_WARPS * 32);
            } else if (rok) {
#pragma unroll
                for (int n = 0; n < NH; ++n) {
                    const int t = ltile * NT + h * NH + n;
                    if (t < Te) a.Y[xe][static_cast<size_t>(t) * a.M + row] = y[n];
                }
            }
        } else {
            // this split's partial sums stay in its shared memory, [NT][MT]
            // (the stages are idle now) for the split-K reduction below
            float *mine = reinterpret_cast<float *>(smem_raw + (stage0 - raw));
#pragma unroll
            for (int n = 0; n < NH; ++n) mine[(h * NH + n) * MT + r] = y[n];
        }
    }
    tc_fence_before();
    if (__syncthreads_or(failed)) {
        // A wait gave up: outputs are unspecified, but nothing this CTA
        // started may land after it exits.  Each producer waits (bounded)
        // for its last copies or MMAs; a completed phase of a barrier
        // implies the earlier ones of the same barrier.
        if (lane == 0 && warp == CODE_WARP) {
            // the last chunk issued into each slot (its full barrier counts
            // only the producer's arrival and the chunk's bytes)
            for (int c = issued > CODE_SLOTS ? issued - CODE_SLOTS : 0; c < issued; ++c)
                mbar_wait_bounded(cfull0 + 8 * (c % CODE_SLOTS), (c / CODE_SLOTS) & 1, nullptr, 0u);
        } else if (lane == 0 && (warp == MMA_WARP || warp == MMA_WARP2) && issued > 0) {
            // the commit of this issuer's last MMA group tracks every
            // earlier one it issued
            const int i = (warp == MMA_WARP ? 0 : 1) + 2 * (issued - 1);
            mbar_wait_bounded(accf0 + 8 * (i % NB), (i / NB) & 1, nullptr, 0u);
        } else if (lane == 0 && warp == BPROD_WARP && issued > 0) {
            // token blocks share their stage's full barrier with the
            // converters' arrivals, which a converter that gave up never
            // makes: give the at most S blocks in flight a bounded time (one
            // block is at most 64 KB; this is about a millisecond)
            const long long t0 = clock64();
            while (clock64() - t0 < 2000000LL) __nanosleep(1000);
        }
        tc_fence_before();
        __syncthreads();
    }

    if (a.nsplit > 1) {
        // ---- split-K: the cluster is the tile's nsplit K splits.  Every
        // thread of every split passes both cluster barriers, whatever its
        // role and whether a wait gave up, so neither can be left waiting.
        cluster_sync();  // every split's partials are in its shared memory
        {
            // every thread of the CTA takes part (the roles are done); each
            // writes outputs, so each first waits for the previous grid
            pdl_wait();
            const int et = threadIdx.x;
            constexpr int NTH = TC_THREADS;
            const int ns = a.nsplit;
            const int q = static_cast<int>(cluster_rank());
            const int n0 = q * NT / ns, n1 = (q + 1) * NT / ns;
            const uint32_t part0 = stage0;  // the same offset in every split
            float *S = reinterpret_cast<float *>(smem_raw + (codes0 - raw));  // [n1 - n0][MT]
            // work item: token n of this rank's columns, 4 consecutive rows;
            // each sum is taken over the splits in split order.  Several
            // items per thread at a time keep U x nsplit remote loads in flight.
            const int items = (n1 - n0) * (MT / 4);
            constexpr int U = 2;
            for (int first = 0; first < items; first += U * NTH) {
                float4 v[U];
#pragma unroll
                for (int u = 0; u < U; ++u) v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int sp = 0; sp < 8; ++sp) {
                    if (sp >= ns) break;  // uniform
                    float4 pv[U];
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int it = first + u * NTH + et;
                        pv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                        if (it < items) {
                            const int n = n0 + (it >> 5), r4 = it & 31;
                            pv[u] = ld_dsmem_f32x4(
                                mapa_shared(part0 + static_cast<uint32_t>(n * MT + 4 * r4) * 4u, sp));
                        }
                    }
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        v[u].x += pv[u].x;
                        v[u].y += pv[u].y;
                        v[u].z += pv[u].z;
                        v[u].w += pv[u].w;
                    }
                }
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int it = first + u * NTH + et;
                    if (it < items)
                        reinterpret_cast<float4 *>(S)[((it >> 5) * MT + 4 * (it & 31)) >> 2] = v[u];
                }
            }
            __syncthreads();
            // this CTA has read every split's partials: it arrives on the
            // closing cluster barrier now and waits on it only before it
            // exits, so the barrier's latency overlaps the finish below
            cluster_arrive();
            if (GU) {
                // SiLU(gate row c) * up row c for the rank's tokens, in place
                for (int it = et; it < (n1 - n0) * 64; it += NTH) {
                    const int n = it >> 6, c = it & 63;
                    float *g = S + n * MT + c;
                    *g = silu_fast(*g) * g[64];
                }
                __syncthreads();
                write_hidden_block<BITS, NT>(a, S, MT, mtile, gtile, ltile, Te, n0, n1, et, NTH);
            } else {
                for (int it = et; it < (n1 - n0) * MT; it += NTH) {
                    const int n = it >> 7, r = it & (MT - 1);
                    const int t = ltile * NT + n0 + n;
                    const int row = mtile * MT + r;
                    if (t < Te && row < a.M) a.Y[xe][static_cast<size_t>(t) * a.M + row] = S[n * MT + r];
                }
            }
        }
        cluster_wait();  // no split leaves while another may still read its partials
    }
    if (!GU && threadIdx.x == 0) pdl_launch_dependents();
    if (warp == MMA_WARP) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(NCOLS) : "memory");
    }
}

// ---------------------------------------------------------------- host side

int pick_nt(int T) { return T > 64 ? 128 : (T > 32 ? 64 : (T > 16 ? 32 : 16)); }

size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

struct GemmPlan {
    int mtiles, kps, nsplit;
};

// Split clusters of a GEMM kernel that can be resident at once (one CTA per
// SM; a cluster's CTAs share a GPC), cached per kernel and cluster size.
template <typename K>
int active_clusters(K kernel, size_t smem, int csize)
{
    static std::mutex mu;
    static std::map<std::pair<const void *, int>, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_pair(reinterpret_cast<const void *>(kernel), csize);
    auto it = cache.find(key);
    if (it == cache.end()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1, 1, static_cast<unsigned>(csize));
        cfg.blockDim = dim3(TC_THREADS);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 1;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = static_cast<unsigned>(csize);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = -1;  // unknown: plan by SM count alone
        }
        it = cache.emplace(key, n).first;
    }
    return it->second;
}

// K splits (at most 8: a split set is one portable cluster) so that the
// tiles' clusters fill about one wave of SMs.
template <typename K>
GemmPlan plan_gemm(K kernel, size_t smem, int mtiles, int ntiles, int nkt, int slots)
{
    GemmPlan p = {mtiles, nkt, 1};
    const int base = mtiles * ntiles;
    int maxs = slots / (base > 0 ? base : 1);
    if (maxs > 8) maxs = 8;
    if (maxs > nkt) maxs = nkt;
    while (maxs > 1) {
        const int fit = active_clusters(kernel, smem, maxs);
        if (fit < 0 || base <= fit) break;
        --maxs;
    }
    if (maxs < 1) maxs = 1;
    p.kps = (nkt + maxs - 1) / maxs;
    p.nsplit = (nkt + p.kps - 1) / p.kps;
    return p;
}

struct TcLayout {
    int nt, ntiles;
    size_t xb, hb, total;
};

// The experts of one grouped launch: up to TC_MAX_EXPERTS with T > 0, their
// first global token tile and one token-tile width for all of them (from
// the largest T).
struct TcGroup {
    int n;
    int idx[TC_MAX_EXPERTS];
    int tile0[TC_MAX_EXPERTS + 1];
    int nt;
};

// Splits experts [0, n) with T > 0 into groups; returns the group count.
int make_groups(int n, const int *T, TcGroup *groups, int max_groups)
{
    int g = 0;
    TcGroup cur = {};
    auto flush = [&]() {
        if (cur.n == 0) return;
        int tmax = 1;
        for (int i = 0; i < cur.n; ++i) tmax = T[cur.idx[i]] > tmax ? T[cur.idx[i]] : tmax;
        cur.nt = pick_nt(tmax);
        cur.tile0[0] = 0;
        for (int i = 0; i < cur.n; ++i) cur.tile0[i + 1] = cur.tile0[i] + (T[cur.idx[i]] + cur.nt - 1) / cur.nt;
        if (g < max_groups) groups[g] = cur;
        ++g;
        cur = TcGroup{};
    };
    for (int e = 0; e < n; ++e) {
        if (T[e] <= 0) continue;
        cur.idx[cur.n++] = e;
        if (cur.n == TC_MAX_EXPERTS) flush();
    }
    flush();
    return g;
}

TcLayout tc_layout_tiles(int ntiles, int nt, int d_model, int d_ff)
{
    TcLayout L = {};
    L.nt = nt;
    L.ntiles = ntiles;
    size_t off = 0;
    L.xb = off; off = align256(off + static_cast<size_t>(L.ntiles) * (d_model / KT) * b_bytes(L.nt));
    L.hb = off; off = align256(off + static_cast<size_t>(L.ntiles) * (d_ff / KT) * b_bytes(L.nt));
    L.total = off;
    return L;
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder()
{
    static EncodeTiled fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(p);
    });
    return fn;
}

// Tensor map of packed codes [rows x K bits / 8 bytes]: boxes of box_rows
// rows x 128 bytes (4 Q4 or 8 Q2 K tiles), 128-byte swizzle, zero fill
// outside the matrix.
bool encode_codes(CUtensorMap *map, const uint8_t *codes, int bits, int rows, int K, int box_rows)
{
    EncodeTiled fn = encoder();
    if (!fn) return false;
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(K) * bits / 8;
    const cuuint64_t dims[2] = {row_bytes, static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(codes), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BITS, int NT, bool GU, bool TWO>
cudaError_t launch_gemm_k(const TcArgs &args, int mtiles, int sms, cudaStream_t stream)
{
    // CTAs per SM: a CTA allocates all 512 TMEM columns (one per SM) or 256
    // (two per SM), and a CTA beyond that would wait in tcgen05.alloc, so
    // shared memory is padded to keep it off: more than half of the SM's
    // 228 KB for one, more than a third for two
    size_t smem = 1024 + CODE_SLOTS * CHUNK_BYTES + static_cast<size_t>(tc_stages(NT, TWO)) * tc_stage_bytes(NT) + 512;
    const size_t pad = TWO ? (80u << 10) : (120u << 10);
    if (smem < pad) smem = pad;
    auto k = tc_ffn<BITS, NT, GU, TWO>;
    cudaError_t e = ensure_dynamic_smem(k, smem);
    if (e != cudaSuccess) return e;
    TcArgs a = args;
    const GemmPlan p = plan_gemm(k, smem, mtiles, a.ntiles, a.K / KT, sms * (TWO ? 2 : 1));
    a.kps = p.kps;
    a.nsplit = p.nsplit;
    return launch_pdl_cluster(k, dim3(mtiles, a.ntiles, a.nsplit), dim3(TC_THREADS), smem, stream,
                              static_cast<unsigned>(a.nsplit), a);
}

template <int BITS, int NT, bool GU>
cudaError_t launch_gemm(const TcArgs &args, int mtiles, int sms, cudaStream_t stream)
{
    if (NT == 16 && mtiles * args.ntiles > sms) return launch_gemm_k<BITS, 16, GU, true>(args, mtiles, sms, stream);
    return launch_gemm_k<BITS, NT, GU, false>(args, mtiles, sms, stream);
}

template <int BITS, bool GU>
cudaError_t launch_gemm_nt(int nt, const TcArgs &a, int mtiles, int sms, cudaStream_t stream)
{
    if (nt == 128) return launch_gemm<BITS, 128, GU>(a, mtiles, sms, stream);
    if (nt == 64) return launch_gemm<BITS, 64, GU>(a, mtiles, sms, stream);
    if (nt == 32) return launch_gemm<BITS, 32, GU>(a, mtiles, sms, stream);
    return launch_gemm<BITS, 16, GU>(a, mtiles, sms, stream);
}

template <bool GU>
cudaError_t launch_gemm_bits(int bits, int nt, const TcArgs &a, int mtiles, int sms, cudaStream_t stream)
{
    return bits == 4 ? launch_gemm_nt<4, GU>(nt, a, mtiles, sms, stream)
                     : launch_gemm_nt<2, GU>(nt, a, mtiles, sms, stream);
}

}  // namespace

bool tc_batch_supported(int T, int d_model, int d_ff, int group)
{
    return T >= 2 && tc_batch_shape_supported(d_model, d_ff, group);
}

bool tc_batch_shape_supported(int d_model, int d_ff, int group)
{
    return group % KT == 0 && d_model % KT == 0 && d_ff % KT == 0 && d_model > 0 && d_ff > 0;
}

size_t tc_batch_workspace_experts(int n, const int *T, int d_model, int d_ff)
{
    const int max_groups = (n + TC_MAX_EXPERTS - 1) / TC_MAX_EXPERTS + 1;
    TcGroup *groups = new TcGroup[max_groups];
    const int ng = make_groups(n, T, groups, max_groups);
    size_t need = 0;
    for (int g = 0; g < ng && g < max_groups; ++g) {
        const size_t t = tc_layout_tiles(groups[g].tile0[groups[g].n], groups[g].nt, d_model, d_ff).total;
        need = t > need ? t : need;
    }
    delete[] groups;
    return need;
}

size_t tc_batch_workspace(int T, int d_model, int d_ff)
{
    return tc_batch_workspace_experts(1, &T, d_model, d_ff);
}

cudaError_t launch_ffn_batch_tc_experts(int bits, int n, const uint8_t *const *gc, const float *const *gs,
                                        const uint8_t *const *uc, const float *const *us,
                                        const uint8_t *const *dc, const float *const *ds,
                                        const float *const *X, float *const *Y, const int *T, int d_model,
                                        int d_ff, int group, void *workspace, cudaStream_t stream)
{
    const DeviceInfo *dev = device_info();
    if (!dev) return cudaErrorInvalidDevice;
    if (!encoder()) return cudaErrorNotSupported;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    unsigned *status = device_status_word();
    // launches go group after group on the stream: a group's token prep
    // waits for the previous group's down projection before it overwrites
    // the shared workspace
    for (int first = 0; first < n;) {
        TcGroup G;
        {
            // the next group: experts first .. with T > 0, at most TC_MAX_EXPERTS
            int last = first, cnt = 0;
            while (last < n && cnt < TC_MAX_EXPERTS) {
                if (T[last] > 0) ++cnt;
                ++last;
            }
            TcGroup tmp[2];
            const int ng = make_groups(last - first, T + first, tmp, 2);
            if (ng == 0) {
                first = last;
                continue;
            }
            G = tmp[0];
            for (int i = 0; i < G.n; ++i) G.idx[i] += first;
            first = last;
        }
        const int ntiles = G.tile0[G.n];
        const TcLayout L = tc_layout_tiles(ntiles, G.nt, d_model, d_ff);

        PrepArgs p = {};
        for (int i = 0; i < G.n; ++i) {
            p.X[i] = X[G.idx[i]];
            p.T[i] = T[G.idx[i]];
        }
        for (int i = 0; i <= G.n; ++i) p.tile0[i] = G.tile0[i];
        p.n = G.n;
        p.bits = bits;
        p.Bblk = ws + L.xb;
        p.K = d_model;
        p.nt = G.nt;
        p.ntiles = ntiles;
        {
            const long long total = static_cast<long long>(ntiles) * G.nt * (d_model / 8);
            long long blocks = (total + 255) / 256;
            const long long cap = static_cast<long long>(dev->sm_count) * 8;
            if (blocks > cap) blocks = cap;
            if (blocks < 1) blocks = 1;
            cudaError_t e = launch_pdl(prep_tokens, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, p);
            if (e != cudaSuccess) return e;
        }

        // TcArgs is ~10 KB: built on the heap, passed by value at launch
        TcArgs *a = new TcArgs();
        TcArgs *b = new TcArgs();
        bool ok = true;
        for (int i = 0; i < G.n && ok; ++i) {
            const int e = G.idx[i];
            ok = encode_codes(&a->tmap[i][0], gc[e], bits, d_ff, d_model, 64) &&
                 encode_codes(&a->tmap[i][1], uc[e], bits, d_ff, d_model, 64) &&
                 encode_codes(&b->tmap[i][0], dc[e], bits, d_model, d_ff, MT);
            b->tmap[i][1] = b->tmap[i][0];
            a->pmap[i] = b->tmap[i][0];
            // scales are prefetched only from a 16-byte aligned start
            a->pscales[i] = (reinterpret_cast<uintptr_t>(ds[e]) & 15u) == 0 ? ds[e] : nullptr;
            a->scales[i][0] = gs[e];
            a->scales[i][1] = us[e];
            b->scales[i][0] = b->scales[i][1] = ds[e];
            a->Y[i] = nullptr;
            b->Y[i] = Y[e];
            a->T[i] = b->T[i] = T[e];
        }
        for (int i = 0; i <= G.n; ++i) a->tile0[i] = b->tile0[i] = G.tile0[i];
        a->n = b->n = G.n;
        a->B = ws + L.xb;
        a->Hb = ws + L.hb;
        a->status = b->status = status;
        a->M = d_ff;
        a->K = d_model;
        a->pM = d_model;
        a->pK = d_ff;
        b->B = ws + L.hb;
        b->Hb = nullptr;
        b->M = d_model;
        b->K = d_ff;
        a->group = b->group = group;
        a->ntiles = b->ntiles = ntiles;
        cudaError_t e = ok ? cudaSuccess : cudaErrorInvalidValue;
        if (e == cudaSuccess) e = launch_gemm_bits<true>(bits, G.nt, *a, d_ff / KT, dev->sm_count, stream);
        if (e == cudaSuccess)
            e = launch_gemm_bits<false>(bits, G.nt, *b, (d_model + MT - 1) / MT, dev->sm_count, stream);
        delete a;
        delete b;
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_ffn_batch_tc(int bits, const uint8_t *const gu_codes[2], const float *const gu_scales[2],
                                const uint8_t *down_codes, const float *down_scales, const float *X, float *Y,
                                int T, int d_model, int d_ff, int group, void *workspace, cudaStream_t stream)
{
    return launch_ffn_batch_tc_experts(bits, 1, &gu_codes[0], &gu_scales[0], &gu_codes[1], &gu_scales[1],
                                       &down_codes, &down_scales, &X, &Y, &T, d_model, d_ff, group, workspace,
                                       stream);
}

}  // namespace smoe
