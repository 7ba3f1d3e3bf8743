/*
 * A plain C99 caller of the library's C ABI (include/sdattn.h), with no
 * Python and no torch: it reads one sparse decode problem from a binary file,
 * runs sparse_decode_attention on the current GPU with the library's own split
 * policy and workspace size, and writes the bf16 output and the device error
 * flags.  tests/test_c_caller_gpu.py builds it with gcc, feeds it seeded
 * workloads and compares its output with the oracle.
 *
 * Input (native byte order): int64 rows, heads, pages, groups, block, R,
 * requests, W, query_len, region_tokens, fp8, gated; float scale, k_scale,
 * v_scale; then query bf16 [rows, heads, 192], cache [pages, groups, block,
 * 384] (bf16, or E4M3 bytes when fp8), regions int32 [rows, R], block_table
 * int32 [requests, W], positions int32 [rows], active uint8 [rows], and when
 * gated the gate bf16 [rows / groups, groups * heads], all dense.  The FP8
 * scales go to the library as device scalars.
 * Output: bf16 [rows, heads, 192], then uint32 device flags.
 * Exit status: 0 on success, else the number of the step that failed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "sdattn.h"

static void *read_bytes(FILE *f, size_t n)
{
    void *p = malloc(n ? n : 1);
    if (p && n && fread(p, 1, n, f) != n) {
        free(p);
        return NULL;
    }
    return p;
}

static void *to_device(const void *host, size_t n)
{
    void *d = NULL;
    if (cudaMalloc(&d, n ? n : 1) != cudaSuccess)
        return NULL;
    if (n && cudaMemcpy(d, host, n, cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(d);
        return NULL;
    }
    return d;
}

/* A dense row-major view. */
static sda_tensor dense(const void *data, int dtype, int ndim, const int64_t *shape)
{
    sda_tensor t;
    int64_t step = 1;
    int i;
    memset(&t, 0, sizeof t);
    t.data = data;
    t.dtype = dtype;
    t.ndim = ndim;
    for (i = ndim - 1; i >= 0; --i) {
        t.shape[i] = shape[i];
        t.stride[i] = step;
        step *= shape[i];
    }
    return t;
}

int main(int argc, char **argv)
{
    int64_t h[12];
    float fs[3];
    FILE *f;
    if (argc != 3)
        return 1;
    f = fopen(argv[1], "rb");
    if (!f || fread(h, sizeof h, 1, f) != 1 || fread(fs, sizeof fs, 1, f) != 1)
        return 2;
    {
        const int64_t rows = h[0], heads = h[1], pages = h[2], groups = h[3], block = h[4], R = h[5];
        const int64_t reqs = h[6], W = h[7], query_len = h[8], region_tokens = h[9], fp8 = h[10], gated = h[11];
        const float scale = fs[0];
        const size_t nq = (size_t)(rows * heads * 192 * 2);
        const size_t nc = (size_t)(pages * groups * block * 384 * (fp8 ? 1 : 2));
        const size_t nr = (size_t)(rows * R * 4), nt = (size_t)(reqs * W * 4), np = (size_t)(rows * 4);
        const size_t na = (size_t)rows, ng = gated ? (size_t)(rows * heads * 2) : 0;
        void *hq = read_bytes(f, nq), *hc = read_bytes(f, nc), *hr = read_bytes(f, nr);
        void *ht = read_bytes(f, nt), *hp = read_bytes(f, np), *ha = read_bytes(f, na);
        void *hg = read_bytes(f, ng);
        void *dq, *dc, *dr, *dt, *dp, *da, *dg = NULL, *dscales = NULL, *dout = NULL, *ws = NULL, *hout;
        const int64_t sq[3] = {rows, heads, 192}, sc[4] = {pages, groups, block, 384};
        const int64_t sr[2] = {rows, R}, st[2] = {reqs, W}, s1[1] = {rows};
        const int64_t sg[2] = {rows / groups, groups * heads};
        sda_tensor q, c, r, t, p, a, o, gt;
        int splits;
        size_t wsb;
        sda_status status;
        uint32_t flags = 0;
        FILE *g;
        fclose(f);
        if (!hq || !hc || !hr || !ht || !hp || !ha || !hg)
            return 3;
        dq = to_device(hq, nq);
        dc = to_device(hc, nc);
        dr = to_device(hr, nr);
        dt = to_device(ht, nt);
        dp = to_device(hp, np);
        da = to_device(ha, na);
        if (!dq || !dc || !dr || !dt || !dp || !da || cudaMalloc(&dout, nq) != cudaSuccess)
            return 4;
        if (gated && !(dg = to_device(hg, ng)))
            return 4;
        if (fp8 && !(dscales = to_device(fs + 1, 2 * sizeof(float))))   /* k_scale, v_scale */
            return 4;
        splits = sparse_decode_splits((int)rows);
        wsb = sparse_decode_workspace_bytes((int)rows, (int)heads, splits);
        if (cudaMalloc(&ws, wsb) != cudaSuccess || cudaMemset(ws, 0, wsb) != cudaSuccess)
            return 5;
        q = dense(dq, SDA_DTYPE_BF16, 3, sq);
        c = dense(dc, fp8 ? SDA_DTYPE_FP8_E4M3 : SDA_DTYPE_BF16, 4, sc);
        r = dense(dr, SDA_DTYPE_INT32, 2, sr);
        t = dense(dt, SDA_DTYPE_INT32, 2, st);
        p = dense(dp, SDA_DTYPE_INT32, 1, s1);
        a = dense(da, SDA_DTYPE_UINT8, 1, s1);
        o = dense(dout, SDA_DTYPE_BF16, 3, sq);
        gt = dense(dg, SDA_DTYPE_BF16, 2, sg);
        status = sparse_decode_attention(&q, &c, &r, &t, &p, &a, &o, scale, (int)query_len, splits,
                                         fp8 ? (const float *)dscales : NULL,
                                         fp8 ? (const float *)dscales + 1 : NULL, gated ? &gt : NULL, 1,
                                         (int)region_tokens, ws, wsb, NULL);
        if (status != SDA_OK) {
            fprintf(stderr, "sparse_decode_attention: %s\n", sparse_decode_status_string(status));
            return 6;
        }
        if (sparse_decode_read_errors(ws, &flags, 0, NULL) != SDA_OK)
            return 7;
        hout = malloc(nq);
        if (!hout || cudaMemcpy(hout, dout, nq, cudaMemcpyDeviceToHost) != cudaSuccess)
            return 8;
        g = fopen(argv[2], "wb");
        if (!g || fwrite(hout, 1, nq, g) != nq || fwrite(&flags, sizeof flags, 1, g) != 1)
            return 9;
        fclose(g);
        printf("splits %d workspace %lu flags %u\n", splits, (unsigned long)wsb, (unsigned)flags);
        cudaFree(dq);
        cudaFree(dc);
        cudaFree(dr);
        cudaFree(dt);
        cudaFree(dp);
        cudaFree(da);
        cudaFree(dout);
        cudaFree(ws);
        cudaFree(dg);
        cudaFree(dscales);
        free(hq);
        free(hc);
        free(hr);
        free(ht);
        free(hp);
        free(ha);
        free(hg);
        free(hout);
    }
    return 0;
}
