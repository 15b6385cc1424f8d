// Ring-step schedule rules shared by the host scheduler and the kernels.
//
// "Ring Attention" glossary page (ultralytics.com/tr), section "Halka Dikkati
// Nasil Calisir": rank i keeps query block i; at step s it holds the key/value
// block that came from the previous rank, j = (i - s) mod N, so N steps pair
// every query block with every key block.  Under a causal mask, ranks holding
// early query blocks skip most key blocks; striped attention gives every rank
// tokens spread evenly along the sequence instead.
//
// With block length L, contiguous rank r holds natural tokens [r L, (r+1) L)
// and striped rank r holds t = a N + r for local index a in [0, L).  For query
// local index a of rank i and key local index b of rank j, the causal rule
// u <= t becomes:
//   contiguous: j < i all keys; j == i keys b <= a; j > i none (block skipped)
//   striped:    j <= i keys b <= a;  j > i keys b < a  (never a whole block)
// Both reduce, per block pair, to "key local index b < limit(a)".
#pragma once

#ifdef __CUDACC__
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

enum {
    RA_CLS_SKIP = 0,       // no visible pair: the block is not visited
    RA_CLS_FULL = 1,       // every pair visible
    RA_CLS_DIAG_INCL = 2,  // visible iff b <= a
    RA_CLS_DIAG_EXCL = 3   // visible iff b <  a
};

// Query and key tiles are 128 tokens along the sequence.
#define RA_TILE 128

// Key block held by rank i at ring step s.
RA_HD int ra_ring_block(int i, int s, int n_blocks)
{
    int j = (i - s) % n_blocks;
    return j < 0 ? j + n_blocks : j;
}

// Class of the block pair (query rank i, key rank j).
RA_HD int ra_block_class(int layout, int causal, int i, int j)
{
    if (!causal)
        return RA_CLS_FULL;
    if (layout == 0)
        return j < i ? RA_CLS_FULL : (j == i ? RA_CLS_DIAG_INCL : RA_CLS_SKIP);
    return j <= i ? RA_CLS_DIAG_INCL : RA_CLS_DIAG_EXCL;
}

// Exclusive bound on the visible key local index for query local index a.
RA_HD int ra_key_limit(int cls, int a, int L)
{
    int lim = 0;
    if (cls == RA_CLS_FULL)
        lim = L;
    else if (cls == RA_CLS_DIAG_INCL)
        lim = a + 1;
    else if (cls == RA_CLS_DIAG_EXCL)
        lim = a;
    return lim < L ? lim : L;
}

// Key tiles of one block a query tile pair visits; ta_max is the larger query
// tile index of the pair, ntiles = ceil(L / RA_TILE).  Diagonal blocks stop at
// the query tile: later key tiles hold no visible key for it.
RA_HD int ra_kv_tiles(int cls, int ta_max, int ntiles)
{
    if (cls == RA_CLS_SKIP)
        return 0;
    if (cls == RA_CLS_FULL)
        return ntiles;
    return ta_max + 1 < ntiles ? ta_max + 1 : ntiles;
}

// One unit of work for the tensor-core kernel: two 128-row query tiles that
// share a kv head and a rank, processed against the same key/value stream.
struct RaUnit {
    int bh0, ta0;   // tile 0: (batch * H + head), query tile index in the rank
    int bh1, ta1;   // tile 1 (equal to tile 0 when absent)
    int rank;       // query rank i
    int cost;       // key tiles visited (scheduling weight)
    int tile1_valid;
    int pad;
};
