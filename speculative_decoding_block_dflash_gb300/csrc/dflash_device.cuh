// Device helpers shared by the attention kernels: key ranges, split chunks,
// page lookups with bounds checks, bf16 conversion.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>

#include "dflash_internal.h"

namespace dflash {

// Visible key positions [lo, hi] (inclusive) of block query i of a request
// with L keys: the block's queries sit at positions L - T + i; causal rows see
// keys up to their own position, a window W > 0 keeps the last W keys ending
// at the query. Empty when hi < lo.
struct KeyRange {
    int32_t lo, hi;
};

__host__ __device__ inline KeyRange row_range(int32_t L, int32_t T, int32_t i, int32_t causal,
                                              int32_t window)
{
    const int32_t p = L - T + i;
    KeyRange r;
    r.hi = causal ? p : L - 1;
    r.lo = 0;
    if (window > 0) {
        r.lo = p - window + 1;
        if (r.lo < 0) r.lo = 0;
    }
    return r;
}

// Key chunk [kb, ke) handled by split c of S for a request of length L (the
// union range of the block, cut at page-size multiples from base).
struct Chunk {
    int32_t kb, ke;
};

__host__ __device__ inline Chunk split_chunk(int32_t L, int32_t T, int32_t window, int32_t page_size,
                                             int32_t S, int32_t c)
{
    int32_t lo = 0;
    if (window > 0) {
        lo = L - T - window + 1;
        if (lo < 0) lo = 0;
    }
    const int32_t base = (lo / page_size) * page_size;
    const int32_t n = L - base;
    int32_t per = (n + S - 1) / S;
    per = ((per + page_size - 1) / page_size) * page_size;
    Chunk ch;
    ch.kb = base + c * per;
    ch.ke = ch.kb + per;
    if (ch.kb < lo) ch.kb = lo;
    if (ch.ke > L) ch.ke = L;
    if (ch.kb > L) ch.kb = L;
    return ch;
}

// seq_len check: L must hold the block and fit the stated bounds.
__device__ inline bool seq_len_ok(const AttnParams& p, int32_t L)
{
    return L >= p.T && L <= p.max_seq_len && L <= p.max_pages * p.page_size;
}

__device__ inline void raise_error(uint32_t* err, uint32_t bits)
{
    if (err) atomicOr(err, bits);
}

// Physical page of key position j of request b, or -1 (and an error bit) when
// the table entry lies outside [0, num_pages).
__device__ inline int32_t lookup_page(const AttnParams& p, int32_t b, int32_t j)
{
    const int32_t page = __ldg(p.page_table + (int64_t)b * p.max_pages + j / p.page_size);
    if (page < 0 || page >= p.num_pages) {
        raise_error(p.err, DFLASH_DEVERR_PAGE_ID);
        return -1;
    }
    return page;
}

__device__ inline float load_elem(const void* base, int64_t idx, int32_t dtype)
{
    if (dtype == DFLASH_BF16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
    return reinterpret_cast<const float*>(base)[idx];
}

__device__ inline void store_elem(void* base, int64_t idx, float v, int32_t dtype)
{
    if (dtype == DFLASH_BF16)
        reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(base)[idx] = v;
}

}  // namespace dflash
