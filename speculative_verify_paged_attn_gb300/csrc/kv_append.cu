// kv_append.cu -- write the new K/V rows of every sequence into its pages.
//
// Semantics ("Speculative Decoding & KV-Cache PagedAttention in Enterprise
// LLM Serving", PagedKVCacheManager.EnsureCapacityAndAppendToken and the
// shared-prefix section; "The Sub-Millisecond Speculative Decoding Meltdown",
// "Custom FP8 Quantized Memory Block Layout"):
//   rows land at positions L .. L+n_new-1 of each sequence; a page past the
//   table's end is taken from the device free stack with count 1; a mapped
//   page whose count is above 1 is cloned first (the shared block loses one
//   reference, the last holder keeps writing in place); FP8 pages carry one
//   fp32 scale per (page, kv head) for K and one for V, rescaled to
//   amax / 448 over the page's history and new rows on every write.
//
// Two launches on the caller's stream:
//   1. append_alloc_kernel, one CTA per sequence: maps, allocates and clones
//      the touched pages and copies the cloned pages (with their scales).
//      Nothing is written into a shared page here, so a clone never reads a
//      page that its last holder is already rewriting.
//   2. append_write_kernel, one CTA per (sequence, touched page): copies the
//      bf16 rows, or requantises the FP8 page (one warp per (kv head, K|V)
//      tile).  It does nothing when the error word is set, so a failed
//      allocation never writes rows into a page that is still shared.
// Both kernels are a few microseconds of HBM traffic: the page copies and row
// writes are 16-byte vector accesses, the FP8 tiles 4-byte groups per lane.
#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kAllocThreads = 128;
constexpr int kWriteThreads = 256;

// Take one block from the top of the free stack, or -1 (error bit raised).
// Only pops run during an append, so a failed pop means the stack was empty.
__device__ int pop_block(const AppendArgs &a) {
    const int old = atomicSub(a.free_top, 1);
    if (old <= 0 || old > a.num_blocks) {
        atomicAdd(a.free_top, 1);
        raise_error(a.err, old <= 0 ? SVPA_DEVERR_FREE_OVERFLOW : SVPA_DEVERR_BAD_VALUE);
        return -1;
    }
    const int blk = a.free_stack[old - 1];
    if (blk < 0 || blk >= a.num_blocks) {
        raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
        return -1;
    }
    return blk;
}

__global__ void __launch_bounds__(kAllocThreads) append_alloc_kernel(const __grid_constant__ AppendArgs a) {
    __shared__ int s_src[kMaxAppendPages], s_dst[kMaxAppendPages];
    __shared__ int s_ncow;
    const int b = blockIdx.x;
    const int L = a.context_lens[b];
    const long long end = (long long)L + a.n_new;
    if (threadIdx.x == 0) s_ncow = 0;
    __syncthreads();
    if (L < 0 || (end + kBlockSize - 1) / kBlockSize > a.max_blocks) {
        if (threadIdx.x == 0) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
        return;
    }
    int32_t *table = a.block_table + (size_t)b * a.max_blocks;
    const int i0 = L / kBlockSize, i1 = (int)((end - 1) / kBlockSize);
    for (int i = i0 + (int)threadIdx.x; i <= i1; i += kAllocThreads) {
        const int e = table[i];
        if (e < 0) {
            if ((long long)i * kBlockSize < L) {  // history without a page
                raise_error(a.err, SVPA_DEVERR_BAD_VALUE);
                continue;
            }
            const int blk = pop_block(a);
            if (blk < 0) continue;
            a.refcount[blk] = 1;
            table[i] = blk;
            continue;
        }
        if (e >= a.num_blocks) {
            raise_error(a.err, SVPA_DEVERR_BAD_BLOCK);
            continue;
        }
        // Each holder in the batch takes one reference away; the one that
        // takes the last is the sole owner left and writes in place.
        const int old = atomicSub(&a.refcount[e], 1);
        if (old <= 1) {
            atomicAdd(&a.refcount[e], 1);
            if (old < 1) raise_error(a.err, SVPA_DEVERR_BAD_VALUE);  // mapped with count 0
            continue;
        }
        const int blk = pop_block(a);
        if (blk < 0) {
            atomicAdd(&a.refcount[e], 1);
            continue;
        }
        a.refcount[blk] = 1;
        table[i] = blk;
        const int slot = atomicAdd(&s_ncow, 1);
        s_src[slot] = e;
        s_dst[slot] = blk;
    }
    __syncthreads();
    const int ncow = s_ncow;
    const size_t words = a.page_bytes / 16;
    for (int c = 0; c < ncow; ++c) {
        const size_t so = (size_t)s_src[c] * words, dof = (size_t)s_dst[c] * words;
        const uint4 *sk = reinterpret_cast<const uint4 *>(a.k_pool) + so;
        const uint4 *sv = reinterpret_cast<const uint4 *>(a.v_pool) + so;
        uint4 *dk = reinterpret_cast<uint4 *>(a.k_pool) + dof;
        uint4 *dv = reinterpret_cast<uint4 *>(a.v_pool) + dof;
        for (size_t w = threadIdx.x; w < words; w += kAllocThreads) {
            const uint4 x = sk[w], y = sv[w];
            dk[w] = x;
            dv[w] = y;
        }
        if (a.fp8)
            for (int h = threadIdx.x; h < a.Hkv; h += kAllocThreads) {
                a.k_scale[(size_t)s_dst[c] * a.Hkv + h] = a.k_scale[(size_t)s_src[c] * a.Hkv + h];
                a.v_scale[(size_t)s_dst[c] * a.Hkv + h] = a.v_scale[(size_t)s_src[c] * a.Hkv + h];
            }
    }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ float f16_bits_to_f32(uint32_t h) {
    float f;
    asm("{\n\t.reg .b16 s;\n\tcvt.u16.u32 s, %1;\n\tcvt.f32.f16 %0, s;\n\t}" : "=f"(f) : "r"(h));
    return f;
}

// Four E4M3 codes (little-endian bytes of w) to their exact values.
__device__ __forceinline__ void decode4(uint32_t w, float (&v)[4]) {
    const uint32_t lo = e4m3x2_to_f16x2(w & 0xffffu), hi = e4m3x2_to_f16x2(w >> 16);
    v[0] = f16_bits_to_f32(lo & 0xffffu);
    v[1] = f16_bits_to_f32(lo >> 16);
    v[2] = f16_bits_to_f32(hi & 0xffffu);
    v[3] = f16_bits_to_f32(hi >> 16);
}

// Round four fp32 values to E4M3 (nearest-even, saturating at +-448).
__device__ __forceinline__ uint32_t encode4(const float (&v)[4]) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(v[1]), "f"(v[0]));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(v[3]), "f"(v[2]));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

__device__ __forceinline__ void load_new4(const uint16_t *row, int d, float (&v)[4]) {
    const uint2 x = *reinterpret_cast<const uint2 *>(row + d);
    v[0] = bf16_bits_to_f32(x.x & 0xffffu);
    v[1] = bf16_bits_to_f32(x.x >> 16);
    v[2] = bf16_bits_to_f32(x.y & 0xffffu);
    v[3] = bf16_bits_to_f32(x.y >> 16);
}

template <bool FP8>
__global__ void __launch_bounds__(kWriteThreads) append_write_kernel(const __grid_constant__ AppendArgs a) {
    if (*reinterpret_cast<volatile int32_t *>(a.err) != 0) return;
    const int b = blockIdx.x;
    const int L = a.context_lens[b];
    const long long end = (long long)L + a.n_new;
    if (L < 0 || (end + kBlockSize - 1) / kBlockSize > a.max_blocks) return;
    const int i = L / kBlockSize + (int)blockIdx.y;
    const long long ps = (long long)i * kBlockSize;
    if (ps >= end) return;
    const int blk = a.block_table[(size_t)b * a.max_blocks + i];
    if (blk < 0 || blk >= a.num_blocks) return;
    const int hist = L > ps ? (L - ps < kBlockSize ? (int)(L - ps) : kBlockSize) : 0;  // history slots
    const int vend = end - ps < kBlockSize ? (int)(end - ps) : kBlockSize;  // slots in use after
    const int D = a.D, Hkv = a.Hkv;
    // source row of page slot s, kv head h: new rows [B, n_new, Hkv, D]
    auto src_row = [&](const uint16_t *src, int s, int h) {
        return src + (((size_t)b * a.n_new + (size_t)(ps + s - L)) * Hkv + h) * D;
    };

    if constexpr (!FP8) {
        const int cpr = D / 8;  // 16-byte chunks per row
        const int nrows = vend - hist;
        const int per_kv = nrows * Hkv * cpr;
        for (int w = threadIdx.x; w < 2 * per_kv; w += kWriteThreads) {
            const int kv = w >= per_kv;
            int r = w - kv * per_kv;
            const int s = hist + r / (Hkv * cpr);
            r %= Hkv * cpr;
            const int h = r / cpr, c = r - h * cpr;
            const uint16_t *src = kv ? a.new_v : a.new_k;
            uint8_t *pool = kv ? a.v_pool : a.k_pool;
            const uint4 x = reinterpret_cast<const uint4 *>(src_row(src, s, h))[c];
            reinterpret_cast<uint4 *>(pool + (((size_t)blk * Hkv + h) * kBlockSize + s) * D * 2)[c] = x;
        }
    } else {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int gpr = D / 4;  // 4-byte groups per row
        const int hist_g = hist * gpr, vend_g = vend * gpr, tile_g = kBlockSize * gpr;
        for (int u = warp; u < 2 * Hkv; u += kWriteThreads / 32) {
            const int kv = u >= Hkv, h = u - kv * Hkv;
            const uint16_t *src = kv ? a.new_v : a.new_k;
            uint32_t *tile = reinterpret_cast<uint32_t *>((kv ? a.v_pool : a.k_pool) +
                                                          ((size_t)blk * Hkv + h) * kBlockSize * D);
            float *scale = (kv ? a.v_scale : a.k_scale) + (size_t)blk * Hkv + h;
            const float old_scale = *scale;
            // amax over the history (code x old scale, one fp32 product) and the new rows
            float amax = 0.f;
            for (int g = lane; g < vend_g; g += 32) {
                float v[4];
                if (g < hist_g) {
                    decode4(tile[g], v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[k] = __fmul_rn(v[k], old_scale);
                } else {
                    const int s = g / gpr;
                    load_new4(src_row(src, s, h), (g - s * gpr) * 4, v);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) amax = fmaxf(amax, fabsf(v[k]));
            }
#pragma unroll
            for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
            const float ns = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
            const bool rescale = hist > 0 && ns != old_scale;
            for (int g = lane; g < tile_g; g += 32) {
                float v[4];
                if (g < hist_g) {
                    if (!rescale) continue;
                    decode4(tile[g], v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[k] = __fdiv_rn(__fmul_rn(v[k], old_scale), ns);
                } else if (g < vend_g) {
                    const int s = g / gpr;
                    load_new4(src_row(src, s, h), (g - s * gpr) * 4, v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) v[k] = __fdiv_rn(v[k], ns);
                } else {
                    tile[g] = 0u;  // slots past the last row
                    continue;
                }
                tile[g] = encode4(v);
            }
            __syncwarp();
            if (lane == 0) *scale = ns;
        }
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream) {
    append_alloc_kernel<<<a.B, kAllocThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const dim3 grid(a.B, (a.n_new + kBlockSize - 1) / kBlockSize + 1);
    if (a.fp8)
        append_write_kernel<true><<<grid, kWriteThreads, 0, stream>>>(a);
    else
        append_write_kernel<false><<<grid, kWriteThreads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace svpa
