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

// Key tiles a unit of rank i visits over ring steps [s_begin, s_end).
RA_HD int ra_unit_cost(int layout, int causal, int i, int ta_max, int ntiles, int n_blocks,
                       int s_begin, int s_end)
{
    int c = 0;
    for (int s = s_begin; s < s_end; ++s)
        c += ra_kv_tiles(ra_block_class(layout, causal, i, ra_ring_block(i, s, n_blocks)), ta_max,
                         ntiles);
    return c;
}

// The units of one launch, enumerated heaviest first without any stored list.
// A unit is (column x, rank i, tile slot y): x runs over pairs of query heads
// of one kv group (group size even: both heads share positions and masks) or
// over single heads (odd group: the unit takes tiles 2y and 2y + 1 of one
// head).  Ranks [i_lo, i_lo + n_act) are active: all of them, except that at
// a single contiguous causal ring step s only ranks i >= s hold a visible
// block, and a space restricted to some ranks (ra_unit_space_ranks) keeps
// only those.
// Order: x fastest; then, when the cost grows with the rank (contiguous
// causal over all steps: cost = i ntiles + tiles of the diagonal block),
// rank descending then tile descending, otherwise tile descending then rank
// descending (the cost depends on the tile only, or on nothing).  Large
// problems put the kv head outermost (see RA_KV_OUTER_ROWS).
struct RaUnitSpace {
    int X, Y;          // columns, tile slots per rank
    int i_lo, n_act;   // active ranks [i_lo, i_lo + n_act)
    int ntiles;        // 128-row tiles per rank block
    int head_pairs;    // 1: two heads per unit; 0: two tiles of one head
    int rank_outer;    // 1: rank-major order; 0: tile-major order
    int H, N, layout, causal, s_begin, s_end;
    int kv_heads;      // B * Hkv
    int kv_outer;      // 1: kv head is the outermost index of the order
};

// Key/value rows (B * Hkv * S) from which the dealing order groups work by kv
// head: below this the K and V of all heads stay in L2 (32K tokens x 8 kv
// heads x d = 128: 134 MB against a 126 MB L2) and a global heaviest-first
// order balances the tail better; from it on (64K tokens x 8 kv heads: 268 MB
// of K and V, 1 GB at 256K) grouping by head keeps L2 reuse.
#define RA_KV_OUTER_ROWS (1ll << 19)

RA_HD RaUnitSpace ra_unit_space(int B, int H, int Hkv, int S, int n_blocks, int layout, int causal,
                                int s_begin, int s_end)
{
    RaUnitSpace sp;
    const int L = S / n_blocks;
    sp.ntiles = (L + RA_TILE - 1) / RA_TILE;
    sp.head_pairs = ((H / Hkv) % 2 == 0) ? 1 : 0;
    sp.X = sp.head_pairs ? B * H / 2 : B * H;
    sp.Y = sp.head_pairs ? sp.ntiles : (sp.ntiles + 1) / 2;
    const bool all_steps = s_begin == 0 && s_end == n_blocks;
    sp.i_lo = (causal && layout == 0 && !all_steps) ? s_begin : 0;
    sp.n_act = n_blocks - sp.i_lo;
    sp.rank_outer = (causal && layout == 0 && all_steps) ? 1 : 0;
    sp.H = H, sp.N = n_blocks, sp.layout = layout, sp.causal = causal;
    sp.s_begin = s_begin, sp.s_end = s_end;
    sp.kv_heads = B * Hkv;
    sp.kv_outer = (long long)B * Hkv * S >= RA_KV_OUTER_ROWS ? 1 : 0;
    return sp;
}

// The same space restricted to ranks [rank_lo, rank_hi): what one device of
// the ring computes (rank_lo + 1 == rank_hi), in the same order and with the
// same costs.
RA_HD RaUnitSpace ra_unit_space_ranks(RaUnitSpace sp, int rank_lo, int rank_hi)
{
    const int lo = sp.i_lo > rank_lo ? sp.i_lo : rank_lo;
    const int hi = sp.i_lo + sp.n_act < rank_hi ? sp.i_lo + sp.n_act : rank_hi;
    sp.i_lo = lo;
    sp.n_act = hi > lo ? hi - lo : 0;
    return sp;
}

RA_HD long long ra_unit_count(const RaUnitSpace &sp)
{
    return (long long)sp.X * sp.n_act * sp.Y;
}

RA_HD RaUnit ra_unit_decode(const RaUnitSpace &sp, long long u)
{
    int x;
    long long r;
    if (sp.kv_outer) {
        // kv head outermost: the CTAs in flight share one kv head's K and V
        // instead of streaming every head's at once
        const int Xg = sp.X / sp.kv_heads;  // columns per kv head
        const long long per_kv = (long long)Xg * sp.n_act * sp.Y;
        const int kvi = (int)(u / per_kv);
        const long long rem = u - kvi * per_kv;
        x = kvi * Xg + (int)(rem % Xg);
        r = rem / Xg;
    } else {
        x = (int)(u % sp.X);
        r = u / sp.X;
    }
    int i, y;
    const int i_top = sp.i_lo + sp.n_act - 1;  // highest active rank
    if (sp.rank_outer) {
        i = i_top - (int)(r / sp.Y);
        y = sp.Y - 1 - (int)(r % sp.Y);
    } else {
        y = sp.Y - 1 - (int)(r / sp.n_act);
        i = i_top - (int)(r % sp.n_act);
    }
    RaUnit U;
    if (sp.head_pairs) {
        const int half = sp.H / 2;
        U.bh0 = (x / half) * sp.H + 2 * (x % half);
        U.bh1 = U.bh0 + 1;
        U.ta0 = U.ta1 = y;
        U.tile1_valid = 1;
    } else {
        U.bh0 = U.bh1 = x;
        U.ta0 = 2 * y;
        U.tile1_valid = 2 * y + 1 < sp.ntiles ? 1 : 0;
        U.ta1 = U.tile1_valid ? 2 * y + 1 : 2 * y;
    }
    U.rank = i;
    U.cost = ra_unit_cost(sp.layout, sp.causal, i, U.ta0 > U.ta1 ? U.ta0 : U.ta1, sp.ntiles, sp.N,
                          sp.s_begin, sp.s_end);
    U.pad = 0;
    return U;
}
