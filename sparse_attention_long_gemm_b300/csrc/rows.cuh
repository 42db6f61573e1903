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

}  // namespace dsa
