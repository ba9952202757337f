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
//   amax / 448 over the page's history and new rows on every write, or one
//   scale per 64-element tile of a row (the implementation checklist's
//   per-64-element block scales), where each new row's tiles are quantised
//   on their own and the history is left as it is.
//
// Two launches on the caller's stream:
//   1. append_alloc_kernel, one CTA per sequence: maps, allocates and clones
//      the touched pages and copies the cloned pages (with their scales).
//      Nothing is written into a shared page here, so a clone never reads a
//      page that its last holder is already rewriting.
//   2. append_write_kernel, one CTA per (sequence, touched page, group of
//      (K|V, kv head) units): copies the bf16 rows, or requantises the FP8
//      tiles (one warp per tile).  It does nothing when the error word is
//      set, so a failed allocation never writes rows into a page that is
//      still shared.  It is a programmatic dependent launch: its CTAs are
//      scheduled while the first kernel runs and wait for its completion.
// The work is a few MB of HBM traffic, so both kernels are latency-bound:
// every access is a 16-byte vector, and each thread issues all its loads
// (4 per thread per round; an FP8 lane holds its whole share of the tile in
// registers) before its stores, so one call costs a few memory round trips.
#include "svpa_device.cuh"
#include "svpa_internal.h"

namespace svpa {

namespace {

constexpr int kAllocThreads = 256;
constexpr int kWriteThreads = 256;
constexpr int kUnitsBf16 = 4;      // (K|V, kv head) row sets per CTA, bf16 pages
constexpr int kMaxChunksFp8 = 8;   // 16-byte chunks per lane: a 16 x 256-byte FP8 tile

constexpr int kLoadsCopy = 4;  // 16-byte loads per thread in flight in a page copy

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
    // the write kernel may be scheduled now; it waits for this grid's completion
    asm volatile("griddepcontrol.launch_dependents;");
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
        for (size_t w0 = threadIdx.x; w0 < words; w0 += (size_t)kLoadsCopy * kAllocThreads) {
            uint4 x[kLoadsCopy], y[kLoadsCopy];
#pragma unroll
            for (int k = 0; k < kLoadsCopy; ++k) {
                const size_t w = w0 + (size_t)k * kAllocThreads;
                if (w < words) {
                    x[k] = sk[w];
                    y[k] = sv[w];
                }
            }
#pragma unroll
            for (int k = 0; k < kLoadsCopy; ++k) {
                const size_t w = w0 + (size_t)k * kAllocThreads;
                if (w < words) {
                    dk[w] = x[k];
                    dv[w] = y[k];
                }
            }
        }
        if (a.fp8) {
            const size_t n = (size_t)a.scales_per_block;
            for (size_t x = threadIdx.x; x < n; x += kAllocThreads) {
                a.k_scale[(size_t)s_dst[c] * n + x] = a.k_scale[(size_t)s_src[c] * n + x];
                a.v_scale[(size_t)s_dst[c] * n + x] = a.v_scale[(size_t)s_src[c] * n + x];
            }
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

// Chunk k (16 bytes) of a work list of n chunks, kLoads per thread in flight:
// every load of a round is issued before its stores.
constexpr int kLoads = 4;

template <bool FP8>
__global__ void __launch_bounds__(kWriteThreads) append_write_kernel(const __grid_constant__ AppendArgs a) {
    // Before the wait only inputs that the allocation kernel never writes are
    // read (lengths, new rows); the table, counts, pages, scales and error
    // word are read after it.
    const int b = blockIdx.x;
    const int L = a.context_lens[b];
    const long long end = (long long)L + a.n_new;
    if (L < 0 || (end + kBlockSize - 1) / kBlockSize > a.max_blocks) return;
    const int i = L / kBlockSize + (int)blockIdx.y;
    const long long ps = (long long)i * kBlockSize;
    if (ps >= end) return;
    const int hist = L > ps ? (L - ps < kBlockSize ? (int)(L - ps) : kBlockSize) : 0;  // history slots
    const int vend = end - ps < kBlockSize ? (int)(end - ps) : kBlockSize;  // slots in use after
    const int D = a.D, Hkv = a.Hkv;
    // source row of page slot s, kv head h: new rows [B, n_new, Hkv, D]
    auto src_row = [&](const uint16_t *src, int s, int h) {
        return src + (((size_t)b * a.n_new + (size_t)(ps + s - L)) * Hkv + h) * D;
    };
    // wait for the allocation kernel; then its block id for this page
    auto wait_block = [&]() -> int {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (*reinterpret_cast<volatile int32_t *>(a.err) != 0) return -1;
        const int blk = a.block_table[(size_t)b * a.max_blocks + i];
        return blk >= 0 && blk < a.num_blocks ? blk : -1;
    };

    if constexpr (!FP8) {
        // this CTA: units u0 .. u0+kUnitsBf16-1 of the 2*Hkv (K|V, kv head) row sets
        const int u0 = (int)blockIdx.z * kUnitsBf16;
        const int units = min(kUnitsBf16, 2 * Hkv - u0);
        const int cpr = D / 8;  // 16-byte chunks per row
        const int nrows = vend - hist;
        const int per_unit = nrows * cpr;
        const int total = units * per_unit;
        // chunk w: unit, page slot and 16-byte column
        auto where = [&](int w, int &u, int &s, int &c) {
            const int uu = w / per_unit;
            const int r = w - uu * per_unit;
            s = hist + r / cpr;
            c = r - (r / cpr) * cpr;
            u = u0 + uu;
        };
        auto load_round = [&](int w0, uint4 (&x)[kLoads]) {
#pragma unroll
            for (int k = 0; k < kLoads; ++k) {
                const int w = w0 + k * kWriteThreads;
                if (w < total) {
                    int u, s, c;
                    where(w, u, s, c);
                    const int kv = u >= Hkv;
                    x[k] = reinterpret_cast<const uint4 *>(src_row(kv ? a.new_v : a.new_k, s, u - kv * Hkv))[c];
                }
            }
        };
        if ((int)threadIdx.x >= total) return;
        uint4 x[kLoads];
        load_round(threadIdx.x, x);  // the first round overlaps the allocation kernel
        const int blk = wait_block();
        if (blk < 0) return;
        for (int w0 = threadIdx.x; w0 < total; w0 += kLoads * kWriteThreads) {
            if (w0 != (int)threadIdx.x) load_round(w0, x);
#pragma unroll
            for (int k = 0; k < kLoads; ++k) {
                const int w = w0 + k * kWriteThreads;
                if (w < total) {
                    int u, s, c;
                    where(w, u, s, c);
                    const int kv = u >= Hkv, h = u - kv * Hkv;
                    reinterpret_cast<uint4 *>((kv ? a.v_pool : a.k_pool) +
                                              (((size_t)blk * Hkv + h) * kBlockSize + s) * D * 2)[c] = x[k];
                }
            }
        }
    } else {
        // one warp per (K|V, kv head) tile of 16 rows x D bytes, in 16-byte chunks
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int u = (int)blockIdx.z * (kWriteThreads / 32) + warp;
        if (u >= 2 * Hkv) return;
        const int kv = u >= Hkv, h = u - kv * Hkv;
        const uint16_t *src = kv ? a.new_v : a.new_k;
        const int cpr = D / 16;  // chunks per row
        const int nch = kBlockSize * cpr;
        // every chunk this lane owns: 16 new bf16 values (loaded before the
        // wait), or 16 history codes (after it)
        uint4 ra[kMaxChunksFp8], rb[kMaxChunksFp8];
#pragma unroll
        for (int k = 0; k < kMaxChunksFp8; ++k) {
            const int c = lane + 32 * k;
            const int s = c / cpr;
            if (c < nch && s >= hist && s < vend) {
                const uint4 *row = reinterpret_cast<const uint4 *>(src_row(src, s, h));
                const int c2 = 2 * (c - s * cpr);
                ra[k] = row[c2];
                rb[k] = row[c2 + 1];
            }
        }
        const int blk = wait_block();
        if (blk < 0) return;
        uint4 *tile = reinterpret_cast<uint4 *>((kv ? a.v_pool : a.k_pool) +
                                                ((size_t)blk * Hkv + h) * kBlockSize * D);
        if (a.scale_tile) {
            // one scale per 64-element tile of a new row (4 chunks, 4
            // consecutive lanes): amax / 448 of its own values; history rows
            // keep codes and scales; codes past the last row are 0
            float *tsc = (kv ? a.v_scale : a.k_scale) + ((size_t)blk * Hkv + h) * kBlockSize * (D / 64);
#pragma unroll
            for (int k = 0; k < kMaxChunksFp8; ++k) {
                const int c = lane + 32 * k;
                if (c >= nch) continue;  // uniform across the warp (nch is a multiple of 32)
                const int s = c / cpr;
                const bool fresh = s >= hist && s < vend;
                const uint32_t w[8] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w, rb[k].x, rb[k].y, rb[k].z, rb[k].w};
                float amax = 0.f;
                if (fresh) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] & 0xffffu)));
                        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] >> 16)));
                    }
                }
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
                amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
                if (s < hist) continue;
                if (!fresh) {
                    tile[c] = make_uint4(0u, 0u, 0u, 0u);
                    continue;
                }
                const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4] = {__fdiv_rn(bf16_bits_to_f32(w[2 * j] & 0xffffu), sc),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j] >> 16), sc),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j + 1] & 0xffffu), sc),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j + 1] >> 16), sc)};
                    o4[j] = encode4(v);
                }
                tile[c] = make_uint4(o4[0], o4[1], o4[2], o4[3]);
                if ((c & 3) == 0) tsc[s * (D / 64) + (c - s * cpr) / 4] = sc;
            }
            return;
        }
        float *scale = (kv ? a.v_scale : a.k_scale) + (size_t)blk * Hkv + h;
        const float old_scale = *scale;
#pragma unroll
        for (int k = 0; k < kMaxChunksFp8; ++k) {
            const int c = lane + 32 * k;
            if (c < nch && c / cpr < hist) ra[k] = tile[c];
        }
        // amax over the history (code x old scale, one fp32 product) and the new rows
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxChunksFp8; ++k) {
            const int c = lane + 32 * k;
            const int s = c / cpr;
            if (!(c < nch && s < vend)) continue;
            const uint32_t w[4] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w};
            if (s < hist) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4];
                    decode4(w[j], v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) amax = fmaxf(amax, fabsf(__fmul_rn(v[e], old_scale)));
                }
            } else {
                const uint32_t w2[4] = {rb[k].x, rb[k].y, rb[k].z, rb[k].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] & 0xffffu)));
                    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[j] >> 16)));
                    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w2[j] & 0xffffu)));
                    amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w2[j] >> 16)));
                }
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float ns = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        const bool rescale = hist > 0 && ns != old_scale;
#pragma unroll
        for (int k = 0; k < kMaxChunksFp8; ++k) {
            const int c = lane + 32 * k;
            if (c >= nch) continue;
            const int s = c / cpr;
            uint4 out = make_uint4(0u, 0u, 0u, 0u);  // slots past the last row
            if (s < hist) {
                if (!rescale) continue;
                const uint32_t w[4] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w};
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4];
                    decode4(w[j], v);
#pragma unroll
                    for (int e = 0; e < 4; ++e) v[e] = __fdiv_rn(__fmul_rn(v[e], old_scale), ns);
                    o4[j] = encode4(v);
                }
                out = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            } else if (s < vend) {
                const uint32_t w[8] = {ra[k].x, ra[k].y, ra[k].z, ra[k].w, rb[k].x, rb[k].y, rb[k].z, rb[k].w};
                uint32_t o4[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    float v[4] = {__fdiv_rn(bf16_bits_to_f32(w[2 * j] & 0xffffu), ns),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j] >> 16), ns),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j + 1] & 0xffffu), ns),
                                  __fdiv_rn(bf16_bits_to_f32(w[2 * j + 1] >> 16), ns)};
                    o4[j] = encode4(v);
                }
                out = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            tile[c] = out;
        }
        __syncwarp();
        if (lane == 0) *scale = ns;
    }
}

}  // namespace

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t stream) {
    append_alloc_kernel<<<a.B, kAllocThreads, 0, stream>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // (sequence, touched page, group of units); launched as a programmatic
    // dependent of the allocation kernel so that its launch overlaps it
    const int units_per_cta = a.fp8 ? kWriteThreads / 32 : kUnitsBf16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.B, (unsigned)((a.n_new + kBlockSize - 1) / kBlockSize + 1),
                       (unsigned)((2 * a.Hkv + units_per_cta - 1) / units_per_cta));
    cfg.blockDim = dim3(kWriteThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.fp8) return cudaLaunchKernelEx(&cfg, append_write_kernel<true>, a);
    return cudaLaunchKernelEx(&cfg, append_write_kernel<false>, a);
}

}  // namespace svpa
