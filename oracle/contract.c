/*
 * Oracle contraction: plain fp64 complex contraction of a tensor network
 * along a given binary tree, by explicit loops.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the bench's CPU
 * baseline load this library; the product path never does.
 *
 * Follows "Crossing the single-GPU memory wall: multi-GPU large-scale tensor
 * network contraction" (digest of arXiv 2606.01852), §1.1: a step A x B -> C
 * keeps the modes of A and B that the two do not share and sums over the
 * shared ones:
 *
 *     C[c] = sum over k of A[c restricted to A, k] * B[c restricted to B, k]
 *
 * No reordering of any kind is done here: every intermediate keeps the
 * "natural" order (A's surviving modes in A's order, then B's surviving
 * modes in B's order), and only the root is permuted to the caller's open
 * order at the very end.  Each output entry is one sum over the summed modes,
 * accumulated in double precision; OpenMP splits the output entries over
 * threads.  Storage is row-major (last listed mode fastest), complex numbers
 * are (re, im) pairs of doubles.
 */
#include <stdlib.h>
#include <string.h>

typedef struct {
    int rank;
    int *modes;
    long long *dims;
    double *data;   /* 2 * size doubles */
    int owned;      /* freed after use when set */
} tens_t;

static long long tsize(const tens_t *t) {
    long long s = 1;
    for (int i = 0; i < t->rank; ++i) s *= t->dims[i];
    return s;
}

/* Row-major stride of mode x in t, or -1 when t does not carry x. */
static long long stride_of(const tens_t *t, int x) {
    long long s = 1;
    for (int i = t->rank - 1; i >= 0; --i) {
        if (t->modes[i] == x) return s;
        s *= t->dims[i];
    }
    return -1;
}

static int has_mode(const tens_t *t, int x) {
    for (int i = 0; i < t->rank; ++i)
        if (t->modes[i] == x) return 1;
    return 0;
}

/* Contract a and b into a freshly allocated tensor in natural order. */
static int contract_pair(const tens_t *a, const tens_t *b, const long long *extents,
                         tens_t *c) {
    int kmodes[128], nk = 0;
    int cmodes[128], nc = 0;
    for (int i = 0; i < a->rank; ++i) {
        if (has_mode(b, a->modes[i])) kmodes[nk++] = a->modes[i];
        else cmodes[nc++] = a->modes[i];
    }
    for (int i = 0; i < b->rank; ++i)
        if (!has_mode(a, b->modes[i])) cmodes[nc++] = b->modes[i];
    if (nc > 128 || nk > 128) return -1;

    c->rank = nc;
    c->modes = (int *)malloc(sizeof(int) * (nc ? nc : 1));
    c->dims = (long long *)malloc(sizeof(long long) * (nc ? nc : 1));
    for (int i = 0; i < nc; ++i) {
        c->modes[i] = cmodes[i];
        c->dims[i] = extents[cmodes[i]];
    }
    long long csize = tsize(c);
    c->data = (double *)calloc((size_t)(2 * csize), sizeof(double));
    c->owned = 1;
    if (!c->data) return -2;

    /* Offsets of every summed-index tuple inside a and b. */
    long long ksize = 1;
    for (int i = 0; i < nk; ++i) ksize *= extents[kmodes[i]];
    long long *koff_a = (long long *)malloc(sizeof(long long) * ksize);
    long long *koff_b = (long long *)malloc(sizeof(long long) * ksize);
    for (long long kk = 0; kk < ksize; ++kk) {
        long long rem = kk, oa = 0, ob = 0;
        for (int i = nk - 1; i >= 0; --i) {
            long long d = extents[kmodes[i]];
            long long v = rem % d;
            rem /= d;
            oa += v * stride_of(a, kmodes[i]);
            ob += v * stride_of(b, kmodes[i]);
        }
        koff_a[kk] = oa;
        koff_b[kk] = ob;
    }
    /* Per output mode: its stride in a (or 0) and in b (or 0). */
    long long sa[128], sb[128];
    for (int i = 0; i < nc; ++i) {
        long long s = stride_of(a, cmodes[i]);
        sa[i] = s < 0 ? 0 : s;
        s = stride_of(b, cmodes[i]);
        sb[i] = s < 0 ? 0 : s;
    }
    const double *A = a->data, *B = b->data;
    double *C = c->data;
#pragma omp parallel for schedule(dynamic, 64)
    for (long long o = 0; o < csize; ++o) {
        long long rem = o, base_a = 0, base_b = 0;
        for (int i = nc - 1; i >= 0; --i) {
            long long d = c->dims[i];
            long long v = rem % d;
            rem /= d;
            base_a += v * sa[i];
            base_b += v * sb[i];
        }
        double re = 0.0, im = 0.0;
        for (long long kk = 0; kk < ksize; ++kk) {
            const double *x = A + 2 * (base_a + koff_a[kk]);
            const double *y = B + 2 * (base_b + koff_b[kk]);
            re += x[0] * y[0] - x[1] * y[1];
            im += x[0] * y[1] + x[1] * y[0];
        }
        C[2 * o] = re;
        C[2 * o + 1] = im;
    }
    free(koff_a);
    free(koff_b);
    return 0;
}

static void release(tens_t *t) {
    free(t->modes);
    free(t->dims);
    if (t->owned) free(t->data);
    t->modes = NULL;
    t->dims = NULL;
    t->data = NULL;
}

/*
 * Contract the whole network.  leaf_modes holds the leaves' mode lists one
 * after the other (ranks[t] entries each); leaf_data[t] points at the leaf's
 * complex entries.  pairs has 2 * n_steps ids in SSA numbering (leaves
 * 0..n-1, step s produces n+s).  out receives the result in open_modes order.
 * Returns 0 on success.
 */
int oracle_contract(int n_leaves, const int *ranks, const int *leaf_modes,
                    const long long *extents, const double *const *leaf_data,
                    int n_steps, const int *pairs, int n_open, const int *open_modes,
                    double *out) {
    int total = n_leaves + n_steps;
    tens_t *ts = (tens_t *)calloc((size_t)(total ? total : 1), sizeof(tens_t));
    const int *mp = leaf_modes;
    for (int t = 0; t < n_leaves; ++t) {
        ts[t].rank = ranks[t];
        ts[t].modes = (int *)malloc(sizeof(int) * (ranks[t] ? ranks[t] : 1));
        ts[t].dims = (long long *)malloc(sizeof(long long) * (ranks[t] ? ranks[t] : 1));
        for (int i = 0; i < ranks[t]; ++i) {
            ts[t].modes[i] = mp[i];
            ts[t].dims[i] = extents[mp[i]];
        }
        mp += ranks[t];
        ts[t].data = (double *)leaf_data[t];
        ts[t].owned = 0;
    }
    int rc = 0;
    for (int s = 0; s < n_steps && rc == 0; ++s) {
        tens_t *a = &ts[pairs[2 * s]], *b = &ts[pairs[2 * s + 1]];
        rc = contract_pair(a, b, extents, &ts[n_leaves + s]);
        release(a);
        release(b);
    }
    if (rc == 0) {
        tens_t *root = &ts[total - 1];
        /* Permute the root from natural order into open_modes order. */
        long long rstride[128];
        long long odims[128];
        for (int i = 0; i < n_open; ++i) {
            rstride[i] = stride_of(root, open_modes[i]);
            odims[i] = extents[open_modes[i]];
            if (rstride[i] < 0) rc = -3;
        }
        if (rc == 0) {
            long long osize = 1;
            for (int i = 0; i < n_open; ++i) osize *= odims[i];
            for (long long o = 0; o < osize; ++o) {
                long long rem = o, src = 0;
                for (int i = n_open - 1; i >= 0; --i) {
                    long long v = rem % odims[i];
                    rem /= odims[i];
                    src += v * rstride[i];
                }
                out[2 * o] = root->data[2 * src];
                out[2 * o + 1] = root->data[2 * src + 1];
            }
        }
    }
    for (int t = 0; t < total; ++t) release(&ts[t]);
    free(ts);
    return rc;
}

/* Threads OpenMP will use (reported by the bench). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
