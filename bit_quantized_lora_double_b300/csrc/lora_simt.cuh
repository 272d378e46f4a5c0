// lora_simt.cuh -- CUDA-core kernels of the LoRA linear layer:
//   k_lora_down     U = P Q^T for a skinny Q (U = X A^T, V = dY B via B^T),
//                   writes bf16 U and bf16 (s * U)
//   k_transpose     B [N, r] -> B^T [r8, N] (zero rows beyond r)
//   k_lora_grad     split-M partial sums of out[j, c] = sum_m P[m, j] Q[m, c]
//   k_grad_reduce   sums the partials in a fixed order, applies s, stores
//                   dA [r, K] or dB [N, r]
//   k_dx_simt       dX = dY W' + (sV) A, NF4 decoded in the N loop
// These serve the backward for M < 64 tokens (and N not a multiple of 8);
// larger M runs on the tcgen05 kernels.
// Sources: xingyuzhitong.com "Fine-Tuning Memory Requirements", sections "LoRA:
// freeze the base, train small adapters" and "QLoRA: quantize the frozen base
// to 4 bits"; inquiringlines.com note, mechanism paragraph.
#pragma once

#include "common.cuh"

namespace qlora {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// U[m, j] = sum_k P[m, k] Q[j, k] (fp32) for j < r: one block of
// kDownThreads per output (m, j), threads striding over K in 8-element
// (16-byte) chunks, then a warp reduction and the warps' sums in warp order.
// Writes U (bf16, stride ldu, may be null) and sU = bf16(s * U) (stride lds);
// the blocks of the outputs (m, j) with r <= j < lds write the zero padding of
// sU. Block 0 also sets zero[0 .. nzero) to 0 (the following kernel's arrival
// counters; zero may be null). Grid: M * lds blocks.
constexpr int kDownThreads = 128;
__global__ void __launch_bounds__(kDownThreads) k_lora_down(const uint16_t *__restrict__ P, int64_t M, int64_t K,
                                                            const uint16_t *__restrict__ Q, int r, float s,
                                                            uint16_t *__restrict__ U, int ldu,
                                                            uint16_t *__restrict__ sU, int lds,
                                                            uint32_t *__restrict__ zero = nullptr, int nzero = 0) {
    // a forward launched as a programmatic dependent may start now; it
    // waits for U before using it
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (zero && blockIdx.x == 0)
        for (int i = threadIdx.x; i < nzero; i += blockDim.x) zero[i] = 0u;
    __shared__ float wsum[kDownThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t o = blockIdx.x;
    const int64_t m = o / lds;
    const int j = (int)(o % lds);
    if (m >= M) return;
    if (j >= r) {
        if (threadIdx.x == 0) sU[m * lds + j] = 0;
        return;
    }
    float acc = 0.0f;
    if ((K & 7) == 0) {
        // rows are 16-byte aligned (the arrays are): 8 elements per load
        const uint4 *pr = reinterpret_cast<const uint4 *>(P + m * K);
        const uint4 *qr = reinterpret_cast<const uint4 *>(Q + (int64_t)j * K);
#pragma unroll 4
        for (int64_t c = threadIdx.x; c < K / 8; c += kDownThreads) {
            const uint4 x = __ldg(pr + c), a = __ldg(qr + c);
            const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, as[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc = fmaf(bf16lo_to_f32(xs[e]), bf16lo_to_f32(as[e]), acc);
                acc = fmaf(bf16hi_to_f32(xs[e]), bf16hi_to_f32(as[e]), acc);
            }
        }
    } else {
        for (int64_t c = threadIdx.x; c < K; c += kDownThreads)
            acc = fmaf(bf16lo_to_f32(P[m * K + c]), bf16lo_to_f32(Q[(int64_t)j * K + c]), acc);
    }
    acc = warp_sum(acc);
    if (lane == 0) wsum[warp] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = wsum[0];
#pragma unroll
        for (int w = 1; w < kDownThreads / 32; ++w) t += wsum[w];
        if (U) U[m * ldu + j] = __bfloat16_as_ushort(__float2bfloat16_rn(t));
        sU[m * lds + j] = __bfloat16_as_ushort(__float2bfloat16_rn(__fmul_rn(s, t)));
    }
}

// out[j, n] = in[n, j] for j < r, 0 for r <= j < r8.
__global__ void k_transpose(const uint16_t *__restrict__ in, int64_t N, int r, int r8, uint16_t *__restrict__ out) {
    const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    for (int j = 0; j < r8; ++j) out[(int64_t)j * N + n] = j < r ? in[n * r + j] : (uint16_t)0;
}

// out[n, j] = in[n, j] for j < r, 0 for r <= j < rp (zero-padded copy, rows of rp).
__global__ void k_pad_cols(const uint16_t *__restrict__ in, int64_t N, int r, int rp, uint16_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= N * rp) return;
    const int64_t n = i / rp;
    const int j = (int)(i % rp);
    out[i] = j < r ? in[n * r + j] : (uint16_t)0;
}

// out [rp, K] = in [r, K] followed by rp - r zero rows.
__global__ void k_pad_rows(const uint16_t *__restrict__ in, int r, int rp, int64_t K, uint16_t *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)rp * K) return;
    out[i] = i < (int64_t)r * K ? in[i] : (uint16_t)0;
}

// Partial sums over one chunk of rows: part[chunk][j][c] = sum_{m in chunk}
// P[m, j] Q[m, c] for c in a 64-column tile, j < r. P is bf16 [M, ldp],
// Q is bf16 [M, C]. Thread layout: 64 columns x 4 j-groups.
__global__ void __launch_bounds__(256) k_lora_grad(const uint16_t *__restrict__ P, int ldp,
                                                   const uint16_t *__restrict__ Q, int64_t M, int64_t C, int r,
                                                   int64_t rows_per_chunk, float *__restrict__ part) {
    __shared__ float sP[64][129];
    const int tc = threadIdx.x & 63, tj = threadIdx.x >> 6;
    const int64_t c = (int64_t)blockIdx.x * 64 + tc;
    const int64_t mbeg = (int64_t)blockIdx.y * rows_per_chunk;
    const int64_t mend = min(M, mbeg + rows_per_chunk);
    const int jper = (r + 3) / 4;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
    for (int64_t mb = mbeg; mb < mend; mb += 64) {
        const int nm = (int)min((int64_t)64, mend - mb);
        __syncthreads();
        for (int i = threadIdx.x; i < nm * r; i += 256) {
            const int mm = i / r, j = i % r;
            sP[mm][j] = bf16lo_to_f32(P[(mb + mm) * ldp + j]);
        }
        __syncthreads();
        for (int mm = 0; mm < nm; ++mm) {
            const float qv = c < C ? bf16lo_to_f32(Q[(mb + mm) * C + c]) : 0.0f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int j = tj * jper + i;
                if (i < jper && j < r) acc[i] = fmaf(sP[mm][j], qv, acc[i]);
            }
        }
    }
    if (c < C) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int j = tj * jper + i;
            if (i < jper && j < r) part[((int64_t)blockIdx.y * r + j) * C + c] = acc[i];
        }
    }
}

// out = s * sum over chunks (in chunk order) of part[chunk][j][c];
// transposed == 0: out[j * C + c] (dA [r, K]); 1: out[c * r + j] (dB [N, r]).
__global__ void k_grad_reduce(const float *__restrict__ part, int nchunks, int r, int64_t C, float s,
                              int transposed, float *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)r * C) return;
    const int64_t j = i / C, c = i % C;
    float acc = 0.0f;
    for (int k = 0; k < nchunks; ++k) acc += part[(int64_t)k * r * C + i];
    const float v = __fmul_rn(s, acc);
    if (transposed) out[c * r + j] = v; else out[i] = v;
}

// ---- tiled SIMT GEMMs with NF4 decode (64 x 64 tiles, 4 x 4 per thread) ---
constexpr int kSt = 64;

// Decodes the 64 codes of block b (row n, columns k0..k0+63 of W') as fp32.
// Thread `half` (0/1) decodes codes 32*half .. 32*half+31.
// (absmax may be null: double-quantized q, s2, mean; tab: level table)
__device__ __forceinline__ void decode_half_block(const uint8_t *__restrict__ codes, const int8_t *__restrict__ q,
                                                  const float *__restrict__ s2, float mean,
                                                  const float *__restrict__ absmax, int tabid, int64_t b, int half,
                                                  float (&f)[32]) {
    const float a = absmax ? absmax[b] : dq_absmax(q[b], s2[b / kGroup], mean);
    const Nf4Table tab = make_table(a, tabid);
    const uint4 cw = reinterpret_cast<const uint4 *>(codes + b * 32)[half];
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t o[4];
        decode8(tab, w[i], o);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[8 * i + 2 * e] = bf16lo_to_f32(o[e]);
            f[8 * i + 2 * e + 1] = bf16hi_to_f32(o[e]);
        }
    }
}

// dX[m, k] = sum_n dY[m, n] W'[n, k] + sum_j sV[m, j] A[j, k]
__global__ void __launch_bounds__(256) k_dx_simt(const uint16_t *__restrict__ dY, int64_t M, int64_t N,
                                                 const uint8_t *__restrict__ codes, const int8_t *__restrict__ q,
                                                 const float *__restrict__ s2, const float *__restrict__ mean_p,
                                                 int64_t K, const uint16_t *__restrict__ sV, int ldv,
                                                 const uint16_t *__restrict__ A, int r, uint16_t *__restrict__ dX,
                                                 const float *__restrict__ absmax, int tab) {
    __shared__ float Ds[kSt][kSt + 1];  // [m][n]
    __shared__ float Ws[kSt][kSt + 1];  // [n][k]
    const int tid = threadIdx.x, tm = tid & 15, tk = tid >> 4;
    const int64_t m0 = (int64_t)blockIdx.y * kSt, k0 = (int64_t)blockIdx.x * kSt;
    const float mean = absmax ? 0.0f : *mean_p;
    float acc[4][4] = {};
    for (int64_t n0 = 0; n0 < N; n0 += kSt) {
        for (int i = tid; i < kSt * kSt; i += 256) {
            const int row = i >> 6, nn = i & 63;
            const int64_t m = m0 + row, n = n0 + nn;
            Ds[row][nn] = (m < M && n < N) ? bf16lo_to_f32(dY[m * N + n]) : 0.0f;
        }
        if (tid < 128) {
            const int row = tid >> 1, half = tid & 1;
            const int64_t n = n0 + row;
            float f[32];
            if (n < N) {
                decode_half_block(codes, q, s2, mean, absmax, tab, (n * K + k0) / kBlock, half, f);
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) f[e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) Ws[row][half * 32 + e] = f[e];
        }
        __syncthreads();
#pragma unroll 8
        for (int nn = 0; nn < kSt; ++nn) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = Ds[tm * 4 + i][nn];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Ws[nn][tk * 4 + j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
    for (int j = 0; j < r; ++j) {
        float v[4], a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int64_t m = m0 + tm * 4 + i;
            v[i] = m < M ? bf16lo_to_f32(sV[m * ldv + j]) : 0.0f;
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) a[jj] = bf16lo_to_f32(A[(int64_t)j * K + k0 + tk * 4 + jj]);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) acc[i][jj] = fmaf(v[i], a[jj], acc[i][jj]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t m = m0 + tm * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) dX[m * K + k0 + tk * 4 + jj] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[i][jj]));
    }
}

// out = bf16(part_0 + part_1 + ... + part_{n-1}) element by element, the sum
// in fp32 in part order; parts are n consecutive bf16 arrays of `count`
// elements (count % 8 == 0, 16-byte aligned). Sums the per-projection dX of a
// projection group on its CUDA-core path.
__global__ void k_sum_parts(const uint16_t *__restrict__ parts, int n, int64_t count, uint16_t *__restrict__ out) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
    if (i >= count) return;
    float acc[8];
    for (int g = 0; g < n; ++g) {
        const uint4 v = *reinterpret_cast<const uint4 *>(parts + (int64_t)g * count + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float x = __uint_as_float((w[e >> 1] >> (16 * (e & 1))) << 16);
            acc[e] = g == 0 ? x : acc[e] + x;
        }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4 *>(out + i) = o;
}

}  // namespace qlora
