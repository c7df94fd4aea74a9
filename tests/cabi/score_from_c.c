/*
 * score_from_c.c -- the C ABI used from plain C, without Python or the CUDA
 * runtime headers: score n frame pairs held in host memory.
 *
 *   score_from_c W H N SEED
 *
 * Frames are 8-bit, filled from a 32-bit linear congruential generator
 * (x = 1664525 x + 1013904223, sample = x >> 24), the reference first, then
 * the distorted frame as the reference plus (x >> 29) - 4, clipped to
 * [0, 255].  Prints one line per frame with the four scores (%.17g), or the
 * library's status message and a non-zero exit code.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "fvif.h"

int main(int argc, char **argv)
{
    if (argc != 5) {
        fprintf(stderr, "usage: %s W H N SEED\n", argv[0]);
        return 2;
    }
    const int w = atoi(argv[1]), h = atoi(argv[2]), n = atoi(argv[3]);
    uint32_t x = (uint32_t)strtoul(argv[4], NULL, 10);
    const size_t npx = (size_t)w * h * (size_t)n;
    unsigned char *ref = malloc(npx), *dist = malloc(npx);
    double *scores = malloc(sizeof(double) * 4 * (size_t)n);
    if (!ref || !dist || !scores)
        return 3;
    for (size_t i = 0; i < npx; ++i) {
        x = 1664525u * x + 1013904223u;
        ref[i] = (unsigned char)(x >> 24);
    }
    for (size_t i = 0; i < npx; ++i) {
        x = 1664525u * x + 1013904223u;
        int v = (int)ref[i] + (int)(x >> 29) - 4;
        dist[i] = (unsigned char)(v < 0 ? 0 : v > 255 ? 255 : v);
    }

    fvif_ctx *ctx = fvif_create(w, h, 8, 1.0f, 2.0);
    if (!ctx) {
        const int st = fvif_last_error(NULL);
        fprintf(stderr, "fvif_create: %s (%d)\n", fvif_strerror(st), st);
        return 1;
    }
    const int st = fvif_score_host(ctx, ref, dist, n, scores);
    if (st != FVIF_OK) {
        fprintf(stderr, "fvif_score_host: %s (%d)\n", fvif_strerror(st), st);
        fvif_destroy(ctx);
        return 1;
    }
    for (int f = 0; f < n; ++f)
        printf("%.17g %.17g %.17g %.17g\n", scores[4 * f], scores[4 * f + 1],
               scores[4 * f + 2], scores[4 * f + 3]);
    fvif_destroy(ctx);
    free(ref);
    free(dist);
    free(scores);
    return 0;
}
