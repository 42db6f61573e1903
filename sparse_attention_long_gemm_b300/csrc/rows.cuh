// rows.cuh -- which keys a query row sees, for packed prefill and decode.
#pragma once

#include "common.cuh"

namespace dsa {

// Where the query of row `r` sits and which key rows it may read.
//   prefill (packed, causal): sequence b with cu[b] <= r < cu[b+1];
//       position t = r - cu[b]; candidate keys are rows cu[b] .. r.
//   decode: row r is sequence r; its n = cache_seqlens[r] cached positions
//       are rows r*max_ctx .. r*max_ctx + n - 1 of the cache; position n-1.
// The checks make every later access stay inside the caller's buffers even
// when the device-side lengths are wrong (the row is then skipped and
// DSA_ERR_DEVICE_DATA raised).
struct RowInfo {
    long long key_base;  // row of position 0 in the key / kv tensors
    int n;               // number of candidate positions (t + 1)
    bool ok;
};

struct RowSpec {
    const int* lens;     // cu_seqlens [batch+1] (prefill) or cache_seqlens [batch] (decode)
    int batch;
    int decode;          // 0 = packed prefill, 1 = decode over caches
    int max_len;         // max_seqlen (prefill) or max_ctx (decode)
    int base;            // decode: sequence index of lens[0] (the indexer runs long batches in
                         // chunks, each with lens pointing at its first sequence); 0 otherwise
    // decode over a paged cache: the caches are pools of num_pages pages of 2^page_log2
    // positions, and position s of sequence b sits in page pages[b * max_pages + s >> page_log2]
    // (page_log2 >= 7, so that a 128-key tile never crosses a page).  nullptr: dense caches,
    // position s of sequence b at row b * max_len + s.
    const int* pages;
    int page_log2;
    int max_pages;
    int num_pages;
};

__device__ __forceinline__ RowInfo row_info(const RowSpec& rs, int r) {
    RowInfo ri;
    if (rs.decode) {
        const int n = __ldg(rs.lens + r);
        ri.key_base = static_cast<long long>(r) * rs.max_len;
        ri.n = n;
        ri.ok = (n >= 1 && n <= rs.max_len);
    } else {
        const int b = find_seq(rs.lens, rs.batch, r);
        const int lo = __ldg(rs.lens + b);
        ri.key_base = lo;
        ri.n = r - lo + 1;
        ri.ok = (lo >= 0 && lo <= r && ri.n <= rs.max_len && __ldg(rs.lens + b + 1) > r);
    }
    if (!ri.ok) {
        ri.n = 0;
        raise_error(DSA_ERR_DEVICE_DATA);
    }
    return ri;
}

// Row of the key / kv pools that holds position s of decode sequence `seq` in a paged cache.
// A page index outside the pool raises DSA_ERR_DEVICE_DATA and reads page 0 instead (an
// in-bounds row).
__device__ __forceinline__ long long key_row_paged(const RowSpec& rs, int seq, int s) {
    int pg = __ldg(rs.pages + static_cast<long long>(seq) * rs.max_pages + (s >> rs.page_log2));
    if (pg < 0 || pg >= rs.num_pages) {
        raise_error(DSA_ERR_DEVICE_DATA);
        pg = 0;
    }
    return (static_cast<long long>(pg) << rs.page_log2) + (s & ((1 << rs.page_log2) - 1));
}
// The same for a cache that may be dense (position s at key_base + s) or paged.
__device__ __forceinline__ long long key_row(const RowSpec& rs, int seq, long long key_base, int s) {
    return rs.pages == nullptr ? key_base + s : key_row_paged(rs, seq, s);
}

}  // namespace dsa
