// Tensor-core (tcgen05) sparse FFN of Q4_0 layers for batches of tokens, with
// the weights dequantised on chip between HBM and the MMAs.
//
// PowerInfer runs its neuron-aware sparse operators on INT4 (Q4_0) models as
// well (de.news.hada.io summary, "Quantisierung und Kompatibilität"): only the
// predicted neurons' rows are read -- here 18 bytes per 32 weights instead of
// 64 -- and multiplied.  The GEMMs are those of pi_mma.cu,
//
//   U[i, t] = W_up[idx_i] . x_hat_t    A = act(U + b)    Y = A^T . W_down^T rows,
//
// on 16-bit tensor-core operands (kind::f16), so every Q4_0 weight is
// dequantised to f16 on its way to the tensor core: w = (q - 8) * s, the
// product of two f16 values rounded once to f16.  A converting thread copies
// its nibbles and scales (cp.async) into its own part of a ring in shared
// memory several steps ahead of their use -- enough bytes in flight to cover
// HBM's latency -- then converts them.  No copy of the weights, dequantised
// or not, goes back to HBM.
//
//   ffn_up_q4    rows of W_up (W_gate) of the CTA's slice of the list, up to
//                128 per pass.  Eight converter warps write each 64-column K
//                step's weights straight into tensor memory (tcgen05.st;
//                warp w: block w / 4 of the step, for the rows of lane quarter
//                w mod 4), where the MMA reads them as its A operand (M = 128
//                rows, N = B rounded up to 16, K = 16 per MMA); warp 9 loads
//                the x_hat tiles (B) into shared memory by TMA; warp 8 issues
//                the MMAs; the epilogue writes A^T as hi and lo f16 parts (as
//                pi_mma.cu does).  ReLU layers run two CTAs per SM.
//   ffn_down_q4  column blocks of 256 x shares of the list.  Eight converter
//                warps, thread t converting neuron t mod 64's 64 columns of
//                atom t / 64 (two Q4_0 blocks) into the 128-byte-swizzled
//                MN-major A tile in shared memory, made visible to the tensor
//                core by fence.proxy.async; warp 9 loads the A^T hi and lo
//                tiles by TMA; warp 8 issues one MMA per K slice and output
//                tile against the hi and lo rows together (N = 2 Np), so the
//                A tile is read once.
//
// Failure handling is that of pi_mma.cu: every wait is bounded and gives up
// on the abort flag; the MMA lane always commits `done`, which every thread
// waits for before tensor memory is read or freed; the TMA lane, the only one
// with asynchronous copies, has barriers of its own and waits for its last
// copies before the CTA exits.  The converting threads wait for their own
// cp.async copies (cp.async.wait_group, which always completes) before they
// leave.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

#include "pi_kernels.h"
#include "pi_tc.cuh"

namespace pi {
namespace {

constexpr int kUpConvW = 8;         // up kernel: warps 0..7 convert (and run the epilogue), 8 MMA, 9 TMA
constexpr int kUpT = 32 * (kUpConvW + 2);
constexpr int kDnConvW = 8;         // down kernel: warps 0..7 convert (and run the epilogue), 8 MMA, 9 TMA
constexpr int kDnT = 32 * (kDnConvW + 2);

// Two f16 weights (q - 8) * s from nibbles of bytes 2j, 2j + 1 of word w (the
// low nibbles, or the high ones): the byte permute puts the two bytes in the
// halves; the nibble masked into the mantissa under the exponent of 1024
// gives 1024 + q or 1024 + 16 q, and an f16-pair subtract (or fma by 1/16 and
// -72) gives q - 8 exactly; the product with the block's scale is rounded
// once to f16.
// an f16 pair given by its bits (a constant needs no conversion at run time)
__device__ __forceinline__ __half2 h2_bits(uint32_t b)
{
    __half2 h;
    memcpy(&h, &b, 4);
    return h;
}

__device__ __forceinline__ uint32_t q4_w2(uint32_t w, int j, bool high, __half2 s2)
{
    const uint32_t t = __byte_perm(w, 0u, j ? 0x4342u : 0x4140u);
    uint32_t m = (t & (high ? 0x00F000F0u : 0x000F000Fu)) | 0x64006400u;
    __half2 x;
    memcpy(&x, &m, 4);
    // 1/16 = 0x2C00, -72 = 0xD480, 1032 = 0x6408 in f16
    x = high ? __hfma2(x, h2_bits(0x2C002C00u), h2_bits(0xD480D480u)) : __hsub2(x, h2_bits(0x64086408u));
    x = __hmul2(x, s2);
    uint32_t o;
    memcpy(&o, &x, 4);
    return o;
}

// The 8 f16 weights of elements e0 .. e0 + 7 (e0 in {0, 8, 16, 24}) of a Q4_0
// block whose 16 nibble bytes are nib and whose scale is s2 (in both halves).
__device__ __forceinline__ uint4 q4_chunk(const uint4 nib, int e0, __half2 s2)
{
    const bool high = e0 >= 16;
    const uint32_t w0 = (e0 & 8) ? nib.z : nib.x, w1 = (e0 & 8) ? nib.w : nib.y;
    return make_uint4(q4_w2(w0, 0, high, s2), q4_w2(w0, 1, high, s2), q4_w2(w1, 0, high, s2),
                      q4_w2(w1, 1, high, s2));
}

__device__ __forceinline__ __half2 scale2(const uint4 sc, int b) // scale b of 8 packed f16
{
    const uint32_t w = b < 4 ? (b < 2 ? sc.x : sc.y) : (b < 6 ? sc.z : sc.w);
    const uint16_t h = (b & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xffffu);
    return __half2half2(__ushort_as_half(h));
}

__device__ __forceinline__ void sts16(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void fence_to_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 16 bytes global -> shared, asynchronous (zero-filled when src_bytes = 0)
__device__ __forceinline__ void cp16(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// 4 bytes global -> shared (L1-allocating form, the one with a 4-byte size)
__device__ __forceinline__ void cp4(uint32_t dst, const void *src, uint32_t src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
template <int N> __device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint4 lds16(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

__device__ __forceinline__ void arrive1(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(b)) : "memory");
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// A converter warp's turn at a tile: every lane waits (bounded) and the warp
// agrees, so that no lane leaves the loop alone.
__device__ __forceinline__ bool warp_wait(uint64_t *b, uint32_t parity, const MmaParams &p)
{
    return __all_sync(~0u, mbar_wait_bounded(b, parity, p));
}

// The warp's writes to a tile are done: each writing lane orders them before
// the tensor core's reads (fence.proxy.async), the warp synchronises, and one
// lane arrives for it.
__device__ __forceinline__ void warp_arrive(uint64_t *b, bool wrote, int lane)
{
    if (wrote) fence_to_async();
    __syncwarp();
    if (lane == 0) arrive1(b);
}


// The raw Q4_0 data a converting thread needs for one 256-column super-stage
// S of its row (two 128-column K steps): the nibbles of blocks 8 S + 4 j +
// 2 h and 8 S + 4 j + 2 h + 1 for j = 0, 1 (its half h of each step) and the
// 16-byte window of the eight scales of blocks 8 S .. 8 S + 7 (the scale part
// of a row is padded to 16 bytes); 80 bytes, zeros for blocks past the row or
// an absent row.  Each thread reads back only what it copied, so
// cp.async.wait_group is all the synchronisation the ring needs.
constexpr uint32_t kUpRaw = 80;

// (any: a valid address that zero-filled copies name instead of an absent row)
__device__ __forceinline__ void copy_half(uint32_t dst, const uint8_t *row, const uint8_t *any, int scB, int S, int h,
                                          int nblk)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gb = 8 * S + 4 * (i >> 1) + 2 * h + (i & 1);
        const bool v = row && gb < nblk;
        cp16(dst + 16u * i, v ? row + scB + (size_t)gb * 16 : any, v ? 16u : 0u);
    }
    const bool v = row && 8 * S < nblk;
    cp16(dst + 64u, v ? row + (size_t)S * 16 : any, v ? 16u : 0u);
}

// 32 columns of this thread's TMEM lane from registers
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
                 "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
                 "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
                 "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D (+)= A . B^T with A (M = 128 rows x K = 16, one row per lane, element
// pairs packed in 32-bit columns) in tensor memory and B in shared memory
__device__ __forceinline__ void mma_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id, uint32_t acc)
{
    asm volatile("{ .reg .pred q; setp.ne.b32 q, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, q; }" ::"r"(
                     d_tmem),
                 "r"(a_tmem), "l"(b), "r"(id), "r"(acc));
}

// 32 f16 pairs: the 64 weights of blocks n0 and n1 (scales s0, s1)
__device__ __forceinline__ void q4_blocks2(const uint4 n0, const uint4 n1, __half2 s0, __half2 s1, uint32_t (&w)[32])
{
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint4 o = q4_chunk(c < 4 ? n0 : n1, 8 * (c & 3), c < 4 ? s0 : s1);
        w[4 * c] = o.x, w[4 * c + 1] = o.y, w[4 * c + 2] = o.z, w[4 * c + 3] = o.w;
    }
}

// up kernel: K step (columns), raw ring depth (super-stages of two steps:
// copies run R - 1 of them ahead), stages, tensor memory, CTAs per SM
constexpr int kUpKS = 128;
template <bool REGLU> struct UpCfg {
    static constexpr int R = 3;
    static constexpr uint32_t raw_slot = 32u * kUpConvW * kUpRaw * (REGLU ? 2u : 1u);
    static constexpr uint32_t T = 3;                          // stages
    static constexpr uint32_t a_col = REGLU ? 128u : 64u;     // first A column (after U [, gate])
    static constexpr uint32_t a_cols = REGLU ? 128u : 64u;    // columns of one A stage (up [, gate])
    static constexpr uint32_t cols = REGLU ? 512u : 256u;     // allocation
    static constexpr int per_sm = REGLU ? 1 : 2;
};

// ------------------------------------------------------------------ up / gate kernel
// The converted weights go to tensor memory, not shared memory: warp w of the
// eight converter warps writes half w / 4 (two Q4_0 blocks) of each
// 128-column K step of the rows in its lane quarter w mod 4, by tcgen05.st,
// into one of T stages; the MMA reads A from there (M = 128 rows, K = 16 per
// MMA, eight per step) and x_hat (B) from the stage's two 64-column tiles in
// shared memory, loaded by TMA onto the same stage barrier.  Local row r of a
// pass sits in TMEM lane 32 (r mod 4) + r / 4, so the rows of a short pass
// spread over all four lane quarters, hence over all four schedulers.
// Tensor memory: U at columns [0, Np), the gate at [64, 64 + Np) (ReGLU), A
// stage s at a_col + s a_cols (up, then gate).  Shared memory: T x_hat stages
// of 2 x Np x 128 bytes; the raw ring (R slots of 256 threads x 80 bytes,
// twice for ReGLU); barriers full[T] (one arrival per converter warp, and the
// TMA lane's with the tiles' bytes), empty[T] (MMA commit), done; the TMEM
// slot; the row ids.
template <bool REGLU>
__global__ void __launch_bounds__(kUpT, UpCfg<REGLU>::per_sm) ffn_up_q4(const __grid_constant__ MmaParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<__half>;
    using C = UpCfg<REGLU>;
    constexpr uint32_t T = C::T;
    const LayerDev &L = *p.layer;
    // the layer's fields in registers: the loops below hold asm with memory
    // clobbers, which would make the compiler read them again every time
    const uint8_t *const Lup = L.up, *const Lgate = L.gate;
    const int upB = L.upB, rowB = L.rowB, scB = L.scB, act_kind = L.act;
    const int *const lidx = p.idx;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    const uint32_t kXs = (uint32_t)Np * 128u, rawoff = T * 2u * kXs;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + rawoff + (size_t)C::R * C::raw_slot);
    uint64_t *empty = full + T;
    uint64_t *done = empty + T;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *sid = reinterpret_cast<int *>(tslot + 4); // [128]
    if (tid == 0) {
        for (uint32_t s = 0; s < T; ++s) mbar_init(full + s, kUpConvW + 1), mbar_init1(empty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const uint32_t tmem = tmem_alloc(tslot, C::cols);
    pdl_enter();
    const int m = list_len(p, n);
    const int s0 = slice_at(m, blockIdx.x, gridDim.x), s1 = slice_at(m, blockIdx.x + 1, gridDim.x);
    const int KT = (d + kUpKS - 1) / kUpKS, nblk = d / 32;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_up = idesc(H::fmt, 0, 0, 128, (uint32_t)Np);
    const int q4 = warp & 3; // the warp's TMEM lane quarter (converters and epilogue)
    uint32_t g = 0, pass = 0; // K steps handled by this thread's role, passes
    bool ok = true;

    for (int r0 = s0; r0 < s1; r0 += 128, ++pass) {
        const int rows = min(128, s1 - r0);
        for (int r = tid; r < 128; r += kUpT) {
            int id = n; // absent: zeros
            if (r < rows) {
                id = lidx ? lidx[r0 + r] : r0 + r;
                if (id < 0 || id >= n) {
                    fail(p, PI_DEV_FLAG);
                    id = n;
                }
            }
            sid[r] = id;
        }
        __syncthreads();
        const uint32_t g0 = g;
        if (warp < kUpConvW) {
            // this thread: local row r, half h of every K step
            const int h = warp >> 2, r = 4 * lane + q4;
            const bool act = r < rows;
            const int id = sid[r];
            const uint8_t *ru = act && id < n ? Lup + (size_t)id * upB : nullptr;
            const uint8_t *rg = REGLU && act && id < n ? Lgate + (size_t)id * rowB : nullptr;
            const uint32_t raw0 = base + rawoff + (uint32_t)tid * kUpRaw * (REGLU ? 2u : 1u);
            const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16) + C::a_col + 32u * (uint32_t)h;
            const int SS = (KT + 1) / 2;
            const auto issue = [&](int q) { // super-stage q into raw slot q mod R, one commit group
                if (q < SS && act) {
                    const uint32_t dst = raw0 + (uint32_t)(q % C::R) * C::raw_slot;
                    copy_half(dst, ru, Lup, scB, q, h, nblk);
                    if (REGLU) copy_half(dst + kUpRaw, rg, Lup, scB, q, h, nblk);
                }
                cp_commit();
            };
            for (int q = 0; q < C::R - 1; ++q) issue(q);
            Cur cs(g, T);
            for (int S = 0; S < SS && ok; ++S) {
                issue(S + C::R - 1);
                cp_wait<C::R - 1>(); // super-stage S has landed (this thread's own copies)
                const uint32_t rs = raw0 + (uint32_t)(S % C::R) * C::raw_slot;
                const uint4 scu = lds16(rs + 64u);
                const uint4 scg = REGLU ? lds16(rs + kUpRaw + 64u) : make_uint4(0, 0, 0, 0);
                for (int j = 0; j < 2 && 2 * S + j < KT; ++j, ++g, cs.next(T)) {
                    if (g >= T && !warp_wait(empty + cs.s, cs.ph ^ 1u, p)) {
                        ok = false;
                        break;
                    }
                    tc_after(); // the MMAs that read this stage are complete
                    // (rows past the pass convert stale data; their lanes are never read)
                    const uint32_t ta = lane_addr + cs.s * C::a_cols;
                    uint32_t w[32];
                    q4_blocks2(lds16(rs + 32u * j), lds16(rs + 32u * j + 16u), scale2(scu, 4 * j + 2 * h),
                               scale2(scu, 4 * j + 2 * h + 1), w);
                    tmem_st32(ta, w);
                    if (REGLU) {
                        q4_blocks2(lds16(rs + kUpRaw + 32u * j), lds16(rs + kUpRaw + 32u * j + 16u),
                                   scale2(scg, 4 * j + 2 * h), scale2(scg, 4 * j + 2 * h + 1), w);
                        tmem_st32(ta + 64u, w);
                    }
                    // the stores are complete and ordered before the MMA lane's reads
                    tmem_st_wait();
                    tc_before();
                    __syncwarp();
                    if (lane == 0) arrive1(full + cs.s);
                }
            }
            cp_wait<0>(); // (none of this thread's copies is left in flight)
        } else if (warp == kUpConvW + 1) {
            if (lane == 0) {
                Cur cs(g, T);
                for (int kt = 0; kt < KT && ok; ++kt, ++g, cs.next(T)) {
                    if (g >= T && !mbar_wait_bounded(empty + cs.s, cs.ph ^ 1u, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t xb = base + cs.s * 2u * kXs;
                    mbar_expect(full + cs.s, 2u * kXs); // (this lane's arrival, with the bytes)
                    tile_load(xb, &p.tm_x, kt * kUpKS, 0, full + cs.s);
                    tile_load(xb + kXs, &p.tm_x, kt * kUpKS + 64, 0, full + cs.s);
                }
            }
        } else if (warp == kUpConvW) {
            if (lane == 0) {
                const uint64_t dX = sdesc(base, 16, 1024); // x_hat stage 0; + byte offset / 16
                Cur cs(g, T);
                for (int kt = 0; kt < KT && ok; ++kt, ++g, cs.next(T)) {
                    if (!mbar_wait_bounded(full + cs.s, cs.ph, p)) {
                        ok = false;
                        break;
                    }
                    tc_after();
                    const uint64_t x = dX + ((cs.s * 2u * kXs) >> 4);
                    const uint32_t a = tmem + C::a_col + cs.s * C::a_cols;
#pragma unroll
                    for (int k = 0; k < kUpKS / 16; ++k) {
                        const uint64_t xk = x + (k < 4 ? 2 * k : (kXs >> 4) + 2 * (k - 4));
                        mma_ta(tmem, a + 8u * k, xk, id_up, (kt | k) != 0);
                        if (REGLU) mma_ta(tmem + 64u, a + 64u + 8u * k, xk, id_up, (kt | k) != 0);
                    }
                    mma_commit(empty + cs.s);
                }
                mma_commit(done); // always: the MMAs issued so far complete before `done` flips
            }
        }
        __syncwarp();
        // every role has handled the pass's KT steps, unless it gave up
        if (ok) g = g0 + (uint32_t)KT;
        const bool settled = mbar_settle(done, pass & 1, p);
        tc_after();
        const bool live = ok && settled && !*(volatile int *)p.abort_flag;
        // epilogue (warps 0..7): lane quarter w mod 4, token chunks of 16
        // alternating between warps w and w + 4; lane l holds local row 4 l + q
        if (warp < kUpConvW) {
            const int r = 4 * lane + q4;
            const int id = sid[r];
            const float bias = id < n ? H::one(*reinterpret_cast<const uint16_t *>(Lup + (size_t)id * upB + rowB)) : 0.f;
            const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
            for (int c0 = 16 * (warp >> 2); c0 < Np; c0 += 32) {
                float u[16], gt[16];
                tmem_ld16(lane_addr + (uint32_t)c0, u);
                if (REGLU) tmem_ld16(lane_addr + 64u + (uint32_t)c0, gt);
                if (r < rows && live) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int t = c0 + jj;
                        if (t < B) {
                            const float rl = fmaxf((REGLU ? gt[jj] : u[jj]) + bias, 0.f);
                            const float a = REGLU ? rl * u[jj] : (act_kind == ACT_SQRELU ? rl * rl : rl);
                            uint16_t hi, lo;
                            split16<H>(id < n ? a : 0.f, hi, lo);
                            p.actT[(size_t)t * p.mstride + r0 + r] = hi;
                            p.actL[(size_t)t * p.mstride + r0 + r] = lo;
                        }
                    }
                }
            }
        }
        tc_before();
        __syncthreads(); // TMEM and sid are reused by the next pass
        tc_after();
    }
    // the list's tail up to a whole 64-neuron step reads as zeros in the down kernel
    if (blockIdx.x == gridDim.x - 1) {
        const int mp = (m + kBK - 1) / kBK * kBK;
        for (int q = tid; q < (mp - m) * B; q += kUpT) {
            const int t = q / (mp - m), i = m + q % (mp - m);
            p.actT[(size_t)t * p.mstride + i] = 0;
            p.actL[(size_t)t * p.mstride + i] = 0;
        }
    }
    // no copy of this CTA may be in flight when it exits: the TMA lane waits
    // for the last round of every stage (bounded, ignoring the abort flag);
    // a stage's round completes only with the TMA lane's own arrival, so
    // converters that gave up leave it incomplete: the TMA lane then waits
    // out the drain limit, which is only ever spent after a failure
    if (warp == kUpConvW + 1 && lane == 0)
        for (uint32_t q = g > T ? g - T : 0u; q < g; ++q) mbar_drain(full + q % T, (q / T) & 1, kDrainNs);
    tmem_free(tmem, C::cols);
}

// ------------------------------------------------------------------ down kernel
// Work unit u = (256-column block cb, share ks of the list), as in pi_mma.cu.
// Per K step of 64 listed neurons the A tile is the neurons' W_down^T columns
// [c0, c0 + 256) in four 64-column MN-major atoms (neuron k's 64 columns of
// atom a: a 128-byte row at a * 8 KB + 128 k, 128-byte swizzle); thread t of
// the eight converter warps converts neuron t mod 64's columns of atom t / 64
// (two Q4_0 blocks), from the raw data it copied (cp.async) kDnR - 1 K steps
// ahead into its own 48 bytes of a ring slot: the two blocks' nibbles, their
// two scales, and the list entry of its neuron kDnR K steps further on (so
// that no list read waits in the step that needs it).  Shared memory: T
// slots of [A 32 KB][A^T hi][A^T lo] (Np x 128 bytes each); the raw ring;
// barriers tfull, xfull, tempty [T], done; the TMEM slot.
constexpr uint32_t kQAtom = 8192;
constexpr int kDnR = 6;           // raw ring depth (K steps)
constexpr uint32_t kDnRaw = 48;   // per thread and K step (40 bytes used)
constexpr uint32_t kDnRawSlot = 32u * kDnConvW * kDnRaw;
__host__ __device__ constexpr uint32_t q4dn_slot(int Np) { return 4 * kQAtom + 2u * (uint32_t)Np * 128u; }
__host__ __device__ constexpr int q4dn_smem(int Np, int T)
{
    return T * (int)q4dn_slot(Np) + kDnR * (int)kDnRawSlot + (3 * T + 1) * 8 + 16;
}

__global__ void __launch_bounds__(kDnT, 1) ffn_down_q4(const __grid_constant__ MmaParams p, int nks, int T)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<__half>;
    const LayerDev &L = *p.layer;
    // the layer's fields in registers (see the up kernel)
    const uint8_t *const Ldn = L.dn;
    const int rowB = L.rowB, scB = L.scB;
    const int *const lidx = p.idx;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    const uint32_t kX = (uint32_t)Np * 128u;
    const uint32_t kSlot = q4dn_slot(Np);
    uint64_t *tfull = reinterpret_cast<uint64_t *>(smem + (size_t)T * kSlot + (size_t)kDnR * kDnRawSlot);
    uint64_t *xfull = tfull + T;
    uint64_t *tempty = xfull + T;
    uint64_t *done = tempty + T;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    if (tid == 0) {
        for (int s = 0; s < T; ++s) mbar_init(tfull + s, kDnConvW), mbar_init1(xfull + s), mbar_init1(tempty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // tile j at columns [2 j Np, 2 (j+1) Np): A . hi^T, then A . lo^T
    const uint32_t tmem = tmem_alloc(tslot, 256);
    pdl_enter();
    const int m = list_len(p, n);
    const int KTall = (m + kBK - 1) / kBK;
    const int ncb = (d + 255) / 256, nblk = d / 32;
    const uint32_t base = smem_addr(smem);
    // one MMA per (k, tile) against the hi and lo rows together (N = 2 Np):
    // the A tile is read once for both
    const uint32_t id_dn = idesc(H::fmt, 1, 0, 128, 2u * (uint32_t)Np);
    uint32_t g = 0, pass = 0;
    bool ok = true;

    for (int u = blockIdx.x; u < ncb * nks; u += gridDim.x, ++pass) {
        const int cb = u / nks, ks = u % nks;
        const int c0 = cb * 256;
        const int k_lo = slice_at(KTall, ks, nks), KT = slice_at(KTall, ks + 1, nks) - k_lo;
        const uint32_t g0 = g;
        if (warp < kDnConvW) {
            const int kn = tid & 63, a = tid >> 6;
            const int bb = c0 / 32 + 2 * a; // this thread's two blocks: bb, bb + 1
            const uint32_t raw0 = base + (uint32_t)T * kSlot + (uint32_t)tid * kDnRaw;
            // the list entry of neuron kn of K step q (n: absent); v: the raw
            // value when it has been read already
            const auto valid = [&](int q) { return q < KT && (k_lo + q) * kBK + kn < m; };
            const auto entry = [&](int q, int v) {
                int id = n;
                if (valid(q)) {
                    id = lidx ? v : (k_lo + q) * kBK + kn;
                    if (id < 0 || id >= n) id = n; // (flagged by the up kernel)
                }
                return id;
            };
            const auto issue = [&](int q, int id) { // K step q into raw slot q mod kDnR, one commit group
                if (q < KT) {
                    const uint32_t dst = raw0 + (uint32_t)(q % kDnR) * kDnRawSlot;
                    const uint8_t *row = id < n ? Ldn + (size_t)id * rowB : nullptr;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const bool v = row && bb + b < nblk;
                        cp16(dst + 16u * b, v ? row + scB + (size_t)(bb + b) * 16 : Ldn, v ? 16u : 0u);
                    }
                    // the scales of blocks bb, bb + 1 (bb is even; the scale part is padded to 16 bytes)
                    const bool v = row && bb < nblk;
                    cp4(dst + 32u, v ? row + (size_t)bb * 2 : Ldn, v ? 4u : 0u);
                    // the list entry of K step q + kDnR
                    const bool e = lidx && valid(q + kDnR);
                    cp4(dst + 36u, e ? (const void *)(lidx + (k_lo + q + kDnR) * kBK + kn) : (const void *)Ldn,
                        e ? 4u : 0u);
                }
                cp_commit();
            };
            for (int q = 0; q < kDnR - 1; ++q) issue(q, entry(q, valid(q) && lidx ? __ldg(lidx + (k_lo + q) * kBK + kn) : 0));
            int idq = entry(kDnR - 1, valid(kDnR - 1) && lidx ? __ldg(lidx + (k_lo + kDnR - 1) * kBK + kn) : 0);
            uint32_t off[8]; // neuron kn's eight 16-byte chunks of atom a in the 128-byte swizzle
#pragma unroll
            for (int c = 0; c < 8; ++c)
                off[c] = (uint32_t)a * kQAtom + (uint32_t)kn * 128u + (((uint32_t)c ^ (uint32_t)(kn & 7)) << 4);
            Cur cs(g, T);
            for (int kt = 0; kt < KT && ok; ++kt, ++g, cs.next(T)) {
                issue(kt + kDnR - 1, idq);
                cp_wait<kDnR - 1>(); // K step kt has landed (this thread's own copies)
                const uint32_t rs = raw0 + (uint32_t)(kt % kDnR) * kDnRawSlot;
                idq = entry(kt + kDnR, (int)lds32(rs + 36u)); // for the next step's copies
                const uint32_t st = cs.s;
                if (g >= (uint32_t)T && !warp_wait(tempty + st, cs.ph ^ 1u, p)) {
                    ok = false;
                    break;
                }
                const uint32_t tb = base + st * kSlot;
                const uint4 nib0 = lds16(rs), nib1 = lds16(rs + 16u);
                const uint32_t sc = lds32(rs + 32u);
                const __half2 s0 = __half2half2(__ushort_as_half((uint16_t)(sc & 0xffffu)));
                const __half2 s1 = __half2half2(__ushort_as_half((uint16_t)(sc >> 16)));
                uint4 o[8];
#pragma unroll
                for (int c = 0; c < 8; ++c) o[c] = q4_chunk(c < 4 ? nib0 : nib1, 8 * (c & 3), c < 4 ? s0 : s1);
#pragma unroll
                for (int c = 0; c < 8; ++c) sts16(tb + off[c], o[c]);
                warp_arrive(tfull + st, true, lane);
            }
            cp_wait<0>(); // (none of this thread's copies is left in flight)
        } else if (warp == kDnConvW + 1) {
            if (lane == 0) {
                Cur cs(g, T);
                for (int kt = 0; kt < KT && ok; ++kt, ++g, cs.next(T)) {
                    const uint32_t st = cs.s;
                    if (g >= (uint32_t)T && !mbar_wait_bounded(tempty + st, cs.ph ^ 1u, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tb = base + st * kSlot;
                    const int k0 = (k_lo + kt) * kBK;
                    mbar_expect(xfull + st, 2u * kX);
                    tile_load(tb + 4 * kQAtom, &p.tm_act, k0, 0, xfull + st);
                    tile_load(tb + 4 * kQAtom + kX, &p.tm_act_lo, k0, 0, xfull + st);
                }
            }
        } else if (warp == kDnConvW) {
            if (lane == 0) {
                // descriptors of slot 0; a byte offset o adds o / 16 (the start address field)
                const uint64_t dA = sdesc(base, kQAtom, 1024), dB = sdesc(base + 4 * kQAtom, 16, 1024);
                Cur cs(g, T);
                for (int kt = 0; kt < KT && ok; ++kt, ++g, cs.next(T)) {
                    const uint32_t st = cs.s;
                    if (!mbar_wait_bounded(tfull + st, cs.ph, p) || !mbar_wait_bounded(xfull + st, cs.ph, p)) {
                        ok = false;
                        break;
                    }
                    tc_after();
                    const uint64_t a0 = dA + ((st * kSlot) >> 4), b = dB + ((st * kSlot) >> 4);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint64_t ad = a0 + (uint64_t)((2 * j * kQAtom + k * 16 * 128) >> 4);
                            mma(tmem + (uint32_t)(2 * j * Np), ad, b + 2 * k, id_dn, (kt | k) != 0);
                        }
                    }
                    mma_commit(tempty + st);
                }
                mma_commit(done);
            }
        }
        __syncwarp();
        if (ok) g = g0 + (uint32_t)KT;
        const bool settled = mbar_settle(done, pass & 1, p);
        tc_after();
        const bool live = ok && settled && !*(volatile int *)p.abort_flag;
        // epilogue: warp w reads TMEM lanes 32 (w mod 4) .. of tile j = w / 4;
        // thread = output column, 16 tokens at a time
        if (warp < kDnConvW) {
            const int j = warp >> 2, q = warp & 3;
            const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
            const int c = c0 + j * 128 + q * 32 + lane;
            const float bd = c < d ? H::one(L.bdown[c]) : 0.f;
            for (int t0 = 0; t0 < Np; t0 += 16) {
                float v[16], vl[16];
                if (KT > 0) {
                    tmem_ld16(lane_addr + (uint32_t)(2 * j * Np + t0), v);
                    tmem_ld16(lane_addr + (uint32_t)(2 * j * Np + Np + t0), vl);
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] += vl[i];
                } else
                    for (int i = 0; i < 16; ++i) v[i] = 0.f;
                if (c < d && live) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int t = t0 + i;
                        if (t < B) {
                            if (nks > 1) p.part[((size_t)ks * B + t) * d + c] = v[i];
                            else if (p.x) p.x[(size_t)t * d + c] += v[i] + bd;
                            else p.y[(size_t)t * d + c] = H::round(v[i] + bd);
                        }
                    }
                }
            }
        }
        tc_before();
        __syncthreads();
        tc_after();
    }
    if (warp == kDnConvW + 1 && lane == 0)
        for (uint32_t q = g > (uint32_t)T ? g - T : 0u; q < g; ++q) mbar_drain(xfull + q % T, (q / T) & 1, kDrainNs);
    tmem_free(tmem, 256);
}

// shared memory one CTA of a kernel may take when `per_sm` of them share an SM
int smem_budget(int per_sm, int optin)
{
    if (per_sm <= 1) return optin;
    int dev = 0, sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
        return 0;
    return std::min(optin, sm / per_sm - 1024); // (1 KB per CTA is reserved by the system)
}

template <bool REGLU>
cudaError_t launch_up_q4(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    using C = UpCfg<REGLU>;
    const int smem = (int)C::T * 2 * p.Npad * 128 + (int)(C::R * C::raw_slot) + (2 * (int)C::T + 1) * 8 + 16 + 128 * 4;
    if (smem > smem_budget(C::per_sm, smem_optin)) return cudaErrorInvalidValue;
    auto kern = ffn_up_q4<REGLU>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid * C::per_sm), dim3(kUpT), smem, s, p);
}

cudaError_t launch_down_q4(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    int T = 4;
    while (T > 2 && q4dn_smem(p.Npad, T) > smem_optin) --T;
    const int smem = q4dn_smem(p.Npad, T);
    if (smem > smem_optin) return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(ffn_down_q4, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // as many shares of the list per 256-column block as keep every SM busy with one unit
    const int ncb = (p.d + 255) / 256;
    const int nks = grid / ncb > 8 ? 8 : (grid / ncb < 1 ? 1 : grid / ncb);
    const int units = ncb * nks;
    e = launch_pdl(ffn_down_q4, dim3(units < grid ? units : grid), dim3(kDnT), smem, s, p, nks, T);
    if (e != cudaSuccess || nks == 1) return e;
    return launch_ffn_merge(p, false, nks, grid, s);
}

} // namespace

cudaError_t launch_ffn_mma_q4(const MmaParams &p, bool reglu, int grid, cudaStream_t s)
{
    int dev = 0, optin = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    e = reglu ? launch_up_q4<true>(p, grid, optin, s) : launch_up_q4<false>(p, grid, optin, s);
    if (e != cudaSuccess) return e;
    return launch_down_q4(p, grid, optin, s);
}

} // namespace pi
