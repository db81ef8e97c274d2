// Tensor-core (tcgen05) sparse FFN of Q4_0 layers for batches of tokens, with
// the weights dequantised in shared memory between HBM and the MMAs.
//
// PowerInfer runs its neuron-aware sparse operators on INT4 (Q4_0) models as
// well (de.news.hada.io summary, "Quantisierung und Kompatibilität"): only the
// predicted neurons' rows are read -- here 18 bytes per 32 weights instead of
// 64 -- and multiplied.  The GEMMs are those of pi_mma.cu,
//
//   U[i, t] = W_up[idx_i] . x_hat_t    A = act(U + b)    Y = A^T . W_down^T rows,
//
// on 16-bit tensor-core operands (kind::f16), so every Q4_0 weight is
// dequantised to f16 on its way into shared memory: w = (q - 8) * s, the
// product of two f16 values rounded once to f16.  The thread that converts a
// row copies its nibbles and scales (cp.async) into a ring in shared memory
// several steps ahead of their use -- enough bytes in flight to cover HBM's
// latency -- then writes the f16 values into the 128-byte-swizzled operand
// tile the MMA reads, makes its writes visible to the tensor core
// (fence.proxy.async) and arrives on the tile's barrier.  No copy of the
// weights, dequantised or not, goes back to HBM.
//
//   ffn_up_q4    rows of W_up (W_gate) of the SM's slice of the list, 128 per
//                pass: thread r of warps 0..3 converts row r, 64 columns per
//                tile; warp 5 loads the x_hat tiles by TMA; warp 4 issues the
//                MMAs (M = 128 rows, N = B rounded up to 16, K = 64 per tile);
//                warps 0..3 run the epilogue, which writes A^T as hi and lo
//                f16 parts (as pi_mma.cu does).
//   ffn_down_q4  column blocks of 256 x shares of the list: thread t converts
//                half of neuron t / 2's 256 columns into the MN-major A tile
//                (four 64-column atoms); warp 5 loads the A^T hi and lo tiles
//                by TMA; the rest as in pi_mma.cu's down kernel.
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

constexpr int kQWarps = 6;          // 0..3 convert (and run the epilogue), 4 MMA, 5 TMA
constexpr int kQT = 32 * kQWarps;
constexpr int kQConv = 128;         // converting threads
constexpr uint32_t kQTile = 16384;  // 128 rows x 64 f16 (K-major, 128-byte swizzle)
constexpr uint32_t kQX = 8192;      // an x_hat tile: up to 64 tokens x 64 columns

// Two f16 weights (q - 8) * s from nibbles of bytes 2j, 2j + 1 of word w (the
// low nibbles, or the high ones): the byte permute puts the two bytes in the
// halves; the nibble masked into the mantissa under the exponent of 1024
// gives 1024 + q or 1024 + 16 q, and an f16-pair subtract (or fma by 1/16 and
// -72) gives q - 8 exactly; the product with the block's scale is rounded
// once to f16.
__device__ __forceinline__ uint32_t q4_w2(uint32_t w, int j, bool high, __half2 s2)
{
    const uint32_t t = __byte_perm(w, 0u, j ? 0x4342u : 0x4140u);
    uint32_t m = (t & (high ? 0x00F000F0u : 0x000F000Fu)) | 0x64006400u;
    __half2 x;
    memcpy(&x, &m, 4);
    x = high ? __hfma2(x, __float2half2_rn(0.0625f), __float2half2_rn(-72.f)) : __hsub2(x, __float2half2_rn(1032.f));
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

// The raw Q4_0 data of one row and one 256-column super-stage S (8 blocks'
// nibbles, then their 8 scales: 144 bytes) copied by the thread that converts
// that row into its own 144 bytes of a ring slot (zeros for blocks past the
// row or an absent row).  Each thread reads back only what it copied, so
// cp.async.wait_group is all the synchronisation the ring needs.
constexpr uint32_t kRawRow = 144;

// (any: a valid address that zero-filled copies name instead of an absent row)
__device__ __forceinline__ void copy_raw(uint32_t dst, const uint8_t *row, const uint8_t *any, int scB, int S,
                                         int nblk)
{
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int gb = 8 * S + b;
        const bool v = row && gb < nblk;
        cp16(dst + 16u * b, v ? row + scB + (size_t)gb * 16 : any, v ? 16u : 0u);
    }
    // scales of blocks 8S .. 8S + 7: 16 bytes at 16 S (the scale part is padded to 16 bytes)
    const bool v = row && 8 * S < nblk;
    cp16(dst + 128u, v ? row + (size_t)S * 16 : any, v ? 16u : 0u);
}

// raw ring depth (super-stages) of the up kernel: copies run R - 1 super-stages ahead
template <bool REGLU> struct UpRing {
    static constexpr int R = REGLU ? 3 : 4;
    static constexpr uint32_t slot = 128u * kRawRow * (REGLU ? 2u : 1u);
};

// ------------------------------------------------------------------ up / gate kernel
// Shared memory: T slots of [A up tile 16 KB][A gate tile 16 KB (ReGLU)][x_hat
// tile 8 KB]; the raw ring (R slots of 128 rows x 144 bytes, and as much for
// the gate rows); barriers tfull[T] (the 128 converting threads), xfull[T]
// (the x_hat tile's bytes), tempty[T] (MMA commit), done; the TMEM slot; the
// row ids.
template <bool REGLU>
__global__ void __launch_bounds__(kQT, 1) ffn_up_q4(const __grid_constant__ MmaParams p, int T)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<__half>;
    const LayerDev &L = *p.layer;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int d = L.d, n = L.n, B = p.B, Np = p.Npad;
    constexpr uint32_t kSlot = kQTile * (REGLU ? 2u : 1u) + kQX;
    using RG = UpRing<REGLU>;
    uint64_t *tfull = reinterpret_cast<uint64_t *>(smem + (size_t)T * kSlot + (size_t)RG::R * RG::slot);
    uint64_t *xfull = tfull + T;
    uint64_t *tempty = xfull + T;
    uint64_t *done = tempty + T;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(done + 1);
    int *sid = reinterpret_cast<int *>(tslot + 4); // [128]
    if (tid == 0) {
        for (int s = 0; s < T; ++s) mbar_init(tfull + s, kQConv), mbar_init1(xfull + s), mbar_init1(tempty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const uint32_t tmem = tmem_alloc(tslot, 256); // U at columns [0, Np), the gate at [2 Np, 3 Np)
    pdl_enter();
    const int m = list_len(p, n);
    const int s0 = slice_at(m, blockIdx.x, gridDim.x), s1 = slice_at(m, blockIdx.x + 1, gridDim.x);
    const int KT = (d + kBK - 1) / kBK, nblk = d / 32;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_up = idesc(H::fmt, 0, 0, 128, (uint32_t)Np);
    uint32_t g = 0, pass = 0; // tiles handled by this thread's role, passes
    bool ok = true;

    for (int r0 = s0; r0 < s1; r0 += 128, ++pass) {
        const int rows = min(128, s1 - r0);
        for (int r = tid; r < 128; r += kQT) {
            int id = n; // absent: zeros
            if (r < rows) {
                id = p.idx ? p.idx[r0 + r] : r0 + r;
                if (id < 0 || id >= n) {
                    fail(p, PI_DEV_FLAG);
                    id = n;
                }
            }
            sid[r] = id;
        }
        __syncthreads();
        const uint32_t g0 = g;
        if (warp < 4) {
            // thread r converts row r: one 64-column tile per K step, from the
            // raw data it copied R - 1 super-stages ahead
            const int r = tid;
            const int id = sid[r];
            const uint8_t *ru = id < n ? L.up + (size_t)id * L.upB : nullptr;
            const uint8_t *rg = REGLU && id < n ? L.gate + (size_t)id * L.rowB : nullptr;
            const uint32_t raw0 = base + (uint32_t)T * kSlot + (uint32_t)r * kRawRow;
            constexpr uint32_t gateOff = 128u * kRawRow;
            const int SS = (KT + 3) / 4;
            const auto issue = [&](int q) { // super-stage q into raw slot q mod R, one commit group
                if (q < SS) {
                    const uint32_t dst = raw0 + (uint32_t)(q % RG::R) * RG::slot;
                    copy_raw(dst, ru, L.up, L.scB, q, nblk);
                    if (REGLU) copy_raw(dst + gateOff, rg, L.up, L.scB, q, nblk);
                }
                cp_commit();
            };
            for (int q = 0; q < RG::R - 1; ++q) issue(q);
            const uint32_t rowoff = (uint32_t)r * 128u, sw = (uint32_t)(r & 7);
            for (int S = 0; S < SS && ok; ++S) {
                issue(S + RG::R - 1);
                cp_wait<RG::R - 1>(); // super-stage S has landed (this thread's own copies)
                const uint32_t rs = raw0 + (uint32_t)(S % RG::R) * RG::slot;
                const uint4 scu = lds16(rs + 128u);
                const uint4 scg = REGLU ? lds16(rs + gateOff + 128u) : make_uint4(0, 0, 0, 0);
                for (int kk = 0; kk < 4 && 4 * S + kk < KT; ++kk, ++g) {
                    const uint32_t st = g % (uint32_t)T;
                    if (g >= (uint32_t)T && !mbar_wait_bounded(tempty + st, ((g / T) - 1) & 1, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tb = base + st * kSlot;
#pragma unroll
                    for (int h = 0; h < 2; ++h) { // the tile's two blocks
                        const int b = 2 * kk + h;
                        const uint4 nu = lds16(rs + 16u * b);
                        const uint4 ng = REGLU ? lds16(rs + gateOff + 16u * b) : make_uint4(0, 0, 0, 0);
                        const __half2 su = scale2(scu, b), sg = scale2(scg, b);
#pragma unroll
                        for (int c4 = 0; c4 < 4; ++c4) {
                            const int c = 4 * h + c4;
                            const uint32_t off = rowoff + (((uint32_t)c ^ sw) << 4);
                            sts16(tb + off, q4_chunk(nu, 8 * c4, su));
                            if (REGLU) sts16(tb + kQTile + off, q4_chunk(ng, 8 * c4, sg));
                        }
                    }
                    fence_to_async();
                    arrive1(tfull + st);
                }
            }
            cp_wait<0>(); // (none of this thread's copies is left in flight)
        } else if (warp == 5) {
            if (lane == 0)
                for (int kt = 0; kt < KT && ok; ++kt, ++g) {
                    const uint32_t st = g % (uint32_t)T;
                    if (g >= (uint32_t)T && !mbar_wait_bounded(tempty + st, ((g / T) - 1) & 1, p)) {
                        ok = false;
                        break;
                    }
                    mbar_expect(xfull + st, (uint32_t)Np * 128u);
                    tile_load(base + st * kSlot + kQTile * (REGLU ? 2u : 1u), &p.tm_x, kt * kBK, 0, xfull + st);
                }
        } else if (warp == 4) {
            if (lane == 0) {
                for (int kt = 0; kt < KT && ok; ++kt, ++g) {
                    const uint32_t st = g % (uint32_t)T, par = (g / T) & 1;
                    if (!mbar_wait_bounded(tfull + st, par, p) || !mbar_wait_bounded(xfull + st, par, p)) {
                        ok = false;
                        break;
                    }
                    tc_after();
                    const uint32_t tb = base + st * kSlot;
                    const uint32_t xb = tb + kQTile * (REGLU ? 2u : 1u);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t bx = sdesc(xb + k * 32, 16, 1024);
                        mma(tmem, sdesc(tb + k * 32, 16, 1024), bx, id_up, (kt | k) != 0);
                        if (REGLU) mma(tmem + (uint32_t)(2 * Np), sdesc(tb + kQTile + k * 32, 16, 1024), bx, id_up, (kt | k) != 0);
                    }
                    mma_commit(tempty + st);
                }
                mma_commit(done); // always: the MMAs issued so far complete before `done` flips
            }
        }
        __syncwarp();
        // every role has handled the pass's KT tiles, unless it gave up
        if (ok) g = g0 + (uint32_t)KT;
        const bool settled = mbar_settle(done, pass & 1, p);
        tc_after();
        const bool live = ok && settled && !*(volatile int *)p.abort_flag;
        // epilogue (warps 0..3): thread = row r (TMEM lane), 16 token columns at a time
        if (warp < 4) {
            const int r = warp * 32 + lane;
            const int id = sid[r];
            const float bias =
                id < n ? H::one(*reinterpret_cast<const uint16_t *>(L.up + (size_t)id * L.upB + L.rowB)) : 0.f;
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
            for (int c0 = 0; c0 < Np; c0 += 16) {
                float u[16], gt[16];
                tmem_ld16(lane_addr + (uint32_t)c0, u);
                if (REGLU) tmem_ld16(lane_addr + (uint32_t)(2 * Np + c0), gt);
                if (r < rows && live) {
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int t = c0 + jj;
                        if (t < B) {
                            const float rl = fmaxf((REGLU ? gt[jj] : u[jj]) + bias, 0.f);
                            const float a = REGLU ? rl * u[jj] : (L.act == ACT_SQRELU ? rl * rl : rl);
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
        for (int q = tid; q < (mp - m) * B; q += kQT) {
            const int t = q / (mp - m), i = m + q % (mp - m);
            p.actT[(size_t)t * p.mstride + i] = 0;
            p.actL[(size_t)t * p.mstride + i] = 0;
        }
    }
    // no copy of this CTA may be in flight when it exits: the TMA lane waits
    // for its last tiles (bounded, ignoring the abort flag)
    if (warp == 5 && lane == 0)
        for (uint32_t q = g > (uint32_t)T ? g - T : 0u; q < g; ++q) mbar_drain(xfull + q % T, (q / T) & 1, kDrainNs);
    tmem_free(tmem, 256);
}

// ------------------------------------------------------------------ down kernel
// Work unit u = (256-column block cb, share ks of the list), as in pi_mma.cu.
// Per K step of 64 listed neurons the A tile is the neurons' W_down^T columns
// [c0, c0 + 256) in four 64-column MN-major atoms (neuron k's 64 columns of
// atom a: a 128-byte row at a * 8 KB + 128 k, 128-byte swizzle); thread t
// converts neuron t / 2's columns c0 + 128 (t & 1) .. + 128 (four Q4_0 blocks,
// two atoms), from the raw data it copied (cp.async) three K steps ahead into
// its own 80 bytes of a ring slot.  Shared memory: T slots of [A 32 KB][A^T
// hi][A^T lo] (Np x 128 bytes each); the raw ring; barriers tfull, xfull,
// tempty [T], done; the TMEM slot.
constexpr uint32_t kQAtom = 8192;
constexpr int kDnR = 4;           // raw ring depth (K steps): copies run 3 K steps ahead
constexpr uint32_t kDnRaw = 80;   // per thread and K step: 4 blocks' nibbles, a 16-byte scale window
constexpr uint32_t kDnRawSlot = 128u * kDnRaw;
__host__ __device__ constexpr uint32_t q4dn_slot(int Np) { return 4 * kQAtom + 2u * (uint32_t)Np * 128u; }
__host__ __device__ constexpr int q4dn_smem(int Np, int T)
{
    return T * (int)q4dn_slot(Np) + kDnR * (int)kDnRawSlot + (3 * T + 1) * 8 + 16;
}

__global__ void __launch_bounds__(kQT, 1) ffn_down_q4(const __grid_constant__ MmaParams p, int nks, int T)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    using H = H16<__half>;
    const LayerDev &L = *p.layer;
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
        for (int s = 0; s < T; ++s) mbar_init(tfull + s, kQConv), mbar_init1(xfull + s), mbar_init1(tempty + s);
        mbar_init1(done);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    const uint32_t tmem = tmem_alloc(tslot, 128); // tile j at columns [j Np, (j+1) Np)
    pdl_enter();
    const int m = list_len(p, n);
    const int KTall = (m + kBK - 1) / kBK;
    const int ncb = (d + 255) / 256, nblk = d / 32;
    const uint32_t base = smem_addr(smem);
    const uint32_t id_dn = idesc(H::fmt, 1, 0, 128, (uint32_t)Np);
    uint32_t g = 0, pass = 0;
    bool ok = true;

    for (int u = blockIdx.x; u < ncb * nks; u += gridDim.x, ++pass) {
        const int cb = u / nks, ks = u % nks;
        const int c0 = cb * 256;
        const int k_lo = slice_at(KTall, ks, nks), KT = slice_at(KTall, ks + 1, nks) - k_lo;
        const uint32_t g0 = g;
        if (warp < 4) {
            const int kn = tid >> 1, h = tid & 1;
            const int bb = (c0 + 128 * h) / 32; // first of this thread's four blocks
            const int bs = bb & ~7;             // first block of the 16-byte scale window
            const uint32_t raw0 = base + (uint32_t)T * kSlot + (uint32_t)tid * kDnRaw;
            // the list entry of neuron kn of K step q (n: absent), one step ahead of its copies
            const auto entry = [&](int q) {
                const int pos = (k_lo + q) * kBK + kn;
                int id = n;
                if (q < KT && pos < m) {
                    id = p.idx ? __ldg(p.idx + pos) : pos;
                    if (id < 0 || id >= n) id = n; // (flagged by the up kernel)
                }
                return id;
            };
            const auto issue = [&](int q, int id) { // K step q into raw slot q mod kDnR, one commit group
                if (q < KT) {
                    const uint32_t dst = raw0 + (uint32_t)(q % kDnR) * kDnRawSlot;
                    const uint8_t *row = id < n ? L.dn + (size_t)id * L.rowB : nullptr;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const bool v = row && bb + b < nblk;
                        cp16(dst + 16u * b, v ? row + L.scB + (size_t)(bb + b) * 16 : L.dn, v ? 16u : 0u);
                    }
                    const bool v = row && bs < nblk;
                    cp16(dst + 64u, v ? row + (size_t)bs * 2 : L.dn, v ? 16u : 0u);
                }
                cp_commit();
            };
            int idq = entry(0);
            for (int q = 0; q < kDnR - 1; ++q) {
                const int nx = entry(q + 1);
                issue(q, idq);
                idq = nx;
            }
            const uint32_t rowoff = (uint32_t)kn * 128u, sw = (uint32_t)(kn & 7);
            for (int kt = 0; kt < KT && ok; ++kt, ++g) {
                const int nx = entry(kt + kDnR); // (its latency passes during this step)
                issue(kt + kDnR - 1, idq);
                idq = nx;
                cp_wait<kDnR - 1>(); // K step kt has landed (this thread's own copies)
                const uint32_t st = g % (uint32_t)T;
                if (g >= (uint32_t)T && !mbar_wait_bounded(tempty + st, ((g / T) - 1) & 1, p)) {
                    ok = false;
                    break;
                }
                const uint32_t tb = base + st * kSlot;
                const uint32_t rs = raw0 + (uint32_t)(kt % kDnR) * kDnRawSlot;
                const uint4 sc = lds16(rs + 64u);
#pragma unroll
                for (int b = 0; b < 4; ++b) { // block b: atom 2h + b / 2, chunks 4 (b & 1) .. + 3
                    const uint4 nib = lds16(rs + 16u * b);
                    const __half2 s2 = scale2(sc, (bb & 4) + b);
                    const uint32_t ab = tb + (uint32_t)(2 * h + (b >> 1)) * kQAtom + rowoff;
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int c = 4 * (b & 1) + c4;
                        sts16(ab + (((uint32_t)c ^ sw) << 4), q4_chunk(nib, 8 * c4, s2));
                    }
                }
                fence_to_async();
                arrive1(tfull + st);
            }
            cp_wait<0>(); // (none of this thread's copies is left in flight)
        } else if (warp == 5) {
            if (lane == 0)
                for (int kt = 0; kt < KT && ok; ++kt, ++g) {
                    const uint32_t st = g % (uint32_t)T;
                    if (g >= (uint32_t)T && !mbar_wait_bounded(tempty + st, ((g / T) - 1) & 1, p)) {
                        ok = false;
                        break;
                    }
                    const uint32_t tb = base + st * kSlot;
                    const int k0 = (k_lo + kt) * kBK;
                    mbar_expect(xfull + st, 2u * kX);
                    tile_load(tb + 4 * kQAtom, &p.tm_act, k0, 0, xfull + st);
                    tile_load(tb + 4 * kQAtom + kX, &p.tm_act_lo, k0, 0, xfull + st);
                }
        } else if (warp == 4) {
            if (lane == 0) {
                for (int kt = 0; kt < KT && ok; ++kt, ++g) {
                    const uint32_t st = g % (uint32_t)T, par = (g / T) & 1;
                    if (!mbar_wait_bounded(tfull + st, par, p) || !mbar_wait_bounded(xfull + st, par, p)) {
                        ok = false;
                        break;
                    }
                    tc_after();
                    const uint32_t tb = base + st * kSlot;
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k) {
                        const uint64_t bh = sdesc(tb + 4 * kQAtom + k * 32, 16, 1024);
                        const uint64_t bl = sdesc(tb + 4 * kQAtom + kX + k * 32, 16, 1024);
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const uint64_t a = sdesc(tb + (uint32_t)(2 * j) * kQAtom + k * 16 * 128, kQAtom, 1024);
                            mma(tmem + (uint32_t)(j * Np), a, bh, id_dn, (kt | k) != 0);
                            mma(tmem + (uint32_t)(j * Np), a, bl, id_dn, 1u);
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
        // epilogue: thread = output column (TMEM lane) of tile j, 16 tokens at a time
        if (warp < 4) {
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
            for (int j = 0; j < 2; ++j) {
                const int c = c0 + j * 128 + warp * 32 + lane;
                const float bd = c < d ? H::one(L.bdown[c]) : 0.f;
                for (int t0 = 0; t0 < Np; t0 += 16) {
                    float v[16];
                    if (KT > 0) tmem_ld16(lane_addr + (uint32_t)(j * Np + t0), v);
                    else
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
        }
        tc_before();
        __syncthreads();
        tc_after();
    }
    if (warp == 5 && lane == 0)
        for (uint32_t q = g > (uint32_t)T ? g - T : 0u; q < g; ++q) mbar_drain(xfull + q % T, (q / T) & 1, kDrainNs);
    tmem_free(tmem, 128);
}

template <bool REGLU>
cudaError_t launch_up_q4(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    constexpr uint32_t slot = kQTile * (REGLU ? 2u : 1u) + kQX;
    const int fixed = (int)(UpRing<REGLU>::R * UpRing<REGLU>::slot) + 16 + 128 * 4;
    int T = 8;
    while (T > 2 && T * (int)slot + (3 * T + 1) * 8 + fixed > smem_optin) --T;
    const int smem = T * (int)slot + (3 * T + 1) * 8 + fixed;
    if (smem > smem_optin) return cudaErrorInvalidValue;
    auto kern = ffn_up_q4<REGLU>;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(grid), dim3(kQT), smem, s, p, T);
}

cudaError_t launch_down_q4(const MmaParams &p, int grid, int smem_optin, cudaStream_t s)
{
    int T = 6;
    while (T > 2 && q4dn_smem(p.Npad, T) > smem_optin) --T;
    const int smem = q4dn_smem(p.Npad, T);
    cudaError_t e = cudaFuncSetAttribute(ffn_down_q4, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // as many shares of the list per 256-column block as keep every SM busy with one unit
    const int ncb = (p.d + 255) / 256;
    const int nks = grid / ncb > 8 ? 8 : (grid / ncb < 1 ? 1 : grid / ncb);
    const int units = ncb * nks;
    e = launch_pdl(ffn_down_q4, dim3(units < grid ? units : grid), dim3(kQT), smem, s, p, nks, T);
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
