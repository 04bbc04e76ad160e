// gdn_chunk_common.cuh -- pieces shared by the two chunked forms of the scan (the
// one-kernel form of gdn_chunked.cu and the two-phase form of gdn_chunked_ws.cu):
// chunk geometry, the bf16 tensor-core operand images in shared memory and their
// hi / lo split, the tensor-memory plan, the per-chunk decay prefix and the Gram
// products. Both forms
// run the same code for these, so they produce the same bits.
#pragma once

#include <cstdint>

#include "gdn_device.cuh"
#include "gdn_tc.cuh"

namespace gdn {
namespace chunk {

constexpr int kC = 32;    // positions per chunk
constexpr int kS = 128;   // state size (dk = dv) of the tensor-core form
constexpr uint32_t kLbo = 128;                 // K-major core matrices: next 8 bf16 of K
constexpr uint32_t kSbo128 = (kS / 8) * 128;   // next 8 rows, K = 128 operands
constexpr uint32_t kSbo32 = (kC / 8) * 128;    // next 8 rows, K = 32 operands

// ---- tensor-core operands in shared memory: bf16 K-major core-matrix images
// (gdn_tc.cuh, 16-bit layout). One 128-row image over K = 128 (dk): rows 0..31
// hi(Gam q), 32..63 hi(W), 64..95 lo(W), 96..127 lo(Gam q); one 160-row image over
// K = 32 (positions) per part: rows 0..127 w_c k_c (by dk), rows 128..159 M (by t),
// hi part then lo part.
constexpr uint32_t kOffWQ = 0;         // the 128-row image
constexpr uint32_t kOffQhi = 0;        //   rows 0..31:   hi(Gam q)
constexpr uint32_t kOffWhi = 8192;     //   rows 32..63:  hi(W)
constexpr uint32_t kOffWlo = 16384;    //   rows 64..95:  lo(W)
constexpr uint32_t kOffQlo = 24576;    //   rows 96..127: lo(Gam q)
constexpr uint32_t kOffKhi = 32768;    // hi part: rows 0..127 hi(w_c k_c)
constexpr uint32_t kOffMhi = 40960;    //          rows 128..159 hi(M)
constexpr uint32_t kOffKlo = 43008;    // lo part: rows 0..127 lo(w_c k_c)
constexpr uint32_t kOffMlo = 51200;    //          rows 128..159 lo(M)
constexpr uint32_t kImgBytes = 53248;

// Raw rows of k and q in shared memory: 528 bytes (132 floats), so row r starts on
// bank 4r and stays float4 aligned.
constexpr uint32_t kRawRow = 528;
constexpr int kRawRowF = kRawRow / 4;
constexpr uint32_t kRawArr = kC * kRawRow;

// ---- tensor memory (columns; lane = dv)
// A tcgen05 bf16 MMA (M = 128, K = 16) costs the tensor pipe about the same for any
// N up to 160, so a chunk takes three groups of MMAs:
//   the S products: hi(S) against the 128-row image (N = 128), then lo(S) against its
//     first 64 rows (N = 64), into the four 32-column blocks of D:
//     D_y = D[kColDyA] + D[kColDyB],   D_u = D[kColDuA] + D[kColDuB];
//   once U is formed (its split into hi(U) at kColUhi and lo(U) at kColUlo), the
//     state update and the rest of y in one N = 160 group against the 160-row image:
//     [S^T | D[kColDyA]] += U^T [w K | M]^T, which needs the accumulator S^T and the
//     D_y block kColDyA side by side.
// hi(S), lo(S) and the parts of U are bf16 pairs, two to a column (gdn_tc.cuh); S^T and
// D are fp32. The parts of U have columns of their own: the two warps that share a
// lane quarter read D_u and write U over different position ranges, and a packed U
// laid over D_u would put one warp's writes on columns the other still reads.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColShi = 0, kColSlo = 64, kColUhi = 128, kColUlo = 160;
constexpr uint32_t kColSacc = 256, kColD = 384;
constexpr uint32_t kColDyA = kColD, kColDuA = kColD + 32, kColDuB = kColD + 64,
                   kColDyB = kColD + 96;
static_assert(kColD + 4 * kC == kTmemCols, "tensor-memory plan fills the allocation");
static_assert(kColSacc + kS == kColDyA, "S^T and the first D_y block are adjacent");
static_assert(kColShi + kS / 2 <= kColSlo && kColSlo + kS / 2 <= kColUhi &&
                  kColUhi + kC / 2 <= kColUlo && kColUlo + kC / 2 <= kColSacc,
              "the packed parts of S and U fit below the accumulator");
static_assert(kOffQhi == kOffWQ && kOffWhi == kOffWQ + 4 * kSbo128 &&
                  kOffWlo == kOffWQ + 8 * kSbo128 && kOffQlo == kOffWQ + 12 * kSbo128,
              "the four 32-row operand images form one 128-row image");
static_assert(kOffKhi == kOffQlo + 4 * kSbo128, "the 160-row images follow the 128-row one");
static_assert(kOffMhi == kOffKhi + 16 * kSbo32 && kOffMlo == kOffKlo + 16 * kSbo32 &&
                  kOffKlo == kOffMhi + 4 * kSbo32 && kOffMlo + 4 * kSbo32 == kImgBytes,
              "w K and M form one 160-row image per part");

__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }

// Named barrier over `count` threads that also ORs `pred` over them: every thread
// gets the same answer, so a role whose warps must stay in step can leave its
// loop together.
__device__ __forceinline__ bool named_barrier_or(int id, int count, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Cumulative log-decay of a chunk from g_lane (lane = position, 0 past the end of
// the sequence): returns gam_lane and sets `last` = gam_31. Every warp that needs
// these runs this same code on the same inputs, so all get the same bits.
__device__ __forceinline__ float chunk_gam_from(float c, int lane, float &last) {
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(FULL_MASK, c, off);
        if (lane >= off) c += o;
    }
    last = __shfl_sync(FULL_MASK, c, 31);
    return c;
}

// One 16-byte unit of an image (8 consecutive K elements of one row) at byte `o` of
// an image whose row groups are `sbo` bytes apart: its row r and first element k0.
__device__ __forceinline__ void image_unit(uint32_t o, uint32_t sbo, int &r, int &k0) {
    r = static_cast<int>((o / sbo) * 8 + (o % 128) / 16);
    k0 = static_cast<int>(((o % sbo) / 128) * 8);
}

// Unit u (0 .. 511) of a w K image part (rows d = dk, K = positions), by the units a
// warp takes: 32 consecutive rows d at one position block cc (8 positions), so that
// the warp's reads of the raw k rows, k[cc + j][d], fall on 32 different banks.
__device__ __forceinline__ void wk_unit(int u, int &d, int &cc) {
    cc = 8 * (u / kS);
    d = u % kS;
}

// x[0..7] split into bf16 hi and lo parts (tc::split_bf16x2, pairs in K order) and
// stored as one 16-byte unit of each part.
__device__ __forceinline__ void split8_store(const float (&x)[8], unsigned char *hi_dst,
                                             unsigned char *lo_dst) {
    uint4 h, l;
    tc::split_bf16x2(x[0], x[1], h.x, l.x);
    tc::split_bf16x2(x[2], x[3], h.y, l.y);
    tc::split_bf16x2(x[4], x[5], h.z, l.z);
    tc::split_bf16x2(x[6], x[7], h.w, l.w);
    *reinterpret_cast<uint4 *>(hi_dst) = h;
    *reinterpret_cast<uint4 *>(lo_dst) = l;
}

// 16 fp32 values of a tensor-memory row split into 8 packed hi and 8 packed lo words.
__device__ __forceinline__ void split16_packed(const float (&x)[16], uint32_t (&hi)[8],
                                               uint32_t (&lo)[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) tc::split_bf16x2(x[2 * e], x[2 * e + 1], hi[e], lo[e]);
}

// The state split of a chunk, for columns c0 .. c0 + NCOL - 1 of the tensor-memory lane
// at trow (one thread's row of S^T): S -> packed (hi, lo), the A operand of the S
// products, and the accumulator scaled to Gam_31 S, ready for the chunk's update; in
// passes of 16 columns. Completes its stores (tcgen05.wait::st) before returning.
template <int NCOL>
__device__ __forceinline__ void split_state_cols(uint32_t trow, int c0, float gn) {
#pragma unroll 1
    for (int h = 0; h < NCOL / 16; ++h) {
        const uint32_t col = c0 + 16 * h;
        uint32_t r[16], hi[8], lo[8];
        tc::tmem_ld16_nowait(trow + kColSacc + col, r);
        tc::tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) tc::split_bf16x2(u2f(r[2 * e]), u2f(r[2 * e + 1]), hi[e], lo[e]);
#pragma unroll
        for (int e = 0; e < 16; ++e) r[e] = f2u(gn * u2f(r[e]));
        tc::tmem_st8(trow + kColShi + col / 2, hi);
        tc::tmem_st8(trow + kColSlo + col / 2, lo);
        tc::tmem_st16(trow + kColSacc + col, r);
    }
    tc::tmem_st_wait();
}

__device__ __forceinline__ void split_state_row(uint32_t trow, int c0, float gn) {
    split_state_cols<64>(trow, c0, gn);
}

// Partial Gram products of row t against columns s0 + 8 j, j < JN, over all of dk:
// kk[j] = k_t . k_s, qk[j] = q_t . k_s. JN is a compile-time count so every load
// of a step is issued before its FMAs.
template <int JN>
__device__ __forceinline__ void gram_row(const float *rk, const float *rq, int t, int s0,
                                         float (&kk)[4], float (&qk)[4]) {
#pragma unroll 2
    for (int i = 0; i < kS; i += 4) {
        const float4 kt = ld4(rk + t * kRawRowF + i), qt = ld4(rq + t * kRawRowF + i);
        float4 ks[JN];
#pragma unroll
        for (int j = 0; j < JN; ++j) ks[j] = ld4(rk + (s0 + 8 * j) * kRawRowF + i);
#pragma unroll
        for (int j = 0; j < JN; ++j) {
            kk[j] = fmaf(kt.x, ks[j].x, kk[j]);
            kk[j] = fmaf(kt.y, ks[j].y, kk[j]);
            kk[j] = fmaf(kt.z, ks[j].z, kk[j]);
            kk[j] = fmaf(kt.w, ks[j].w, kk[j]);
            qk[j] = fmaf(qt.x, ks[j].x, qk[j]);
            qk[j] = fmaf(qt.y, ks[j].y, qk[j]);
            qk[j] = fmaf(qt.z, ks[j].z, qk[j]);
            qk[j] = fmaf(qt.w, ks[j].w, qk[j]);
        }
    }
}

// The Gram products of a chunk by the 256 threads of 8 warps (gw = 0..7): thread
// (gw, lane) takes row t = 4 rb + lane / 8 against columns s = s0 + 8 j, s0 = lane % 8,
// j < 4, and returns kk[j] = k_t . k_s, qk[j] = q_t . k_s for the blocks j that reach
// the lower triangle (0 for the others). Warps gw and gw + 4 share an SM
// sub-partition, so a short row block is paired with a long one (0+7, 2+5, 1+6, 3+4).
__device__ __forceinline__ void gram_products(const float *rk, const float *rq, int gw, int lane,
                                              int &t, int &s0, float (&kk)[4], float (&qk)[4]) {
    const int pb = gw & 3, rb0 = ((pb & 1) << 1) | (pb >> 1);
    const int rb = gw < 4 ? rb0 : 7 - rb0;
    t = 4 * rb + (lane >> 3);
    s0 = lane & 7;
    const int jmax = (4 * rb + 3) >> 3;  // last block j with 8 j <= the warp's max t
#pragma unroll
    for (int j = 0; j < 4; ++j) kk[j] = qk[j] = 0.f;
    switch (jmax) {  // warp-uniform
        case 0: gram_row<1>(rk, rq, t, s0, kk, qk); break;
        case 1: gram_row<2>(rk, rq, t, s0, kk, qk); break;
        case 2: gram_row<3>(rk, rq, t, s0, kk, qk); break;
        default: gram_row<4>(rk, rq, t, s0, kk, qk); break;
    }
}

}  // namespace chunk
}  // namespace gdn
