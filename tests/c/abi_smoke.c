/* Plain C99 use of the C ABI: the header compiles as C, the shared library links and
 * its host-only calls answer as documented (no GPU is touched). Exit status 0 when
 * every check passes; each failure prints one line. */
#include <stdio.h>
#include <string.h>

#include "splitkv.h"

static int fails = 0;
#define CHECK(cond)                                          \
    do {                                                     \
        if (!(cond)) {                                       \
            printf("FAILED line %d: %s\n", __LINE__, #cond); \
            ++fails;                                         \
        }                                                    \
    } while (0)

static size_t a256(size_t x) { return (x + 255u) & ~(size_t)255u; }

int main(void) {
    sk_params p;
    int s = -1;
    size_t bytes = 0;

    CHECK(sk_version() > 0);
    CHECK(sk_status_string(SK_OK) != NULL && strlen(sk_status_string(SK_ERR_WORKSPACE)) > 0);
    CHECK(sk_supported_head_dims(192, 128) == 1);
    CHECK(sk_supported_head_dims(128, 128) == 1);
    CHECK(sk_supported_head_dims(96, 64) == 0);
    CHECK(sk_default_block_m(192, 128, SK_BF16) == 256);

    /* the target shape: 16 M blocks x 12 heads <= 2 x 152 SMs and 42700 >= 8192 keys */
    memset(&p, 0, sizeof p);
    p.B = 1;
    p.H = 12;
    p.max_seqlen_q = p.total_q = 4096;
    p.max_seqlen_k = p.total_k = 42700;
    p.d_qk = 192;
    p.d_v = 128;
    p.mask = SK_MASK_NONE;
    p.last_valid_kv_index = -1;
    p.n_per_block = 128;
    p.split_kv = 0;
    p.window_left = -1;
    CHECK(sk_choose_split_kv(&p, 152, &s) == SK_OK && s == 3);
    p.max_seqlen_k = p.total_k = 8191; /* below the 8192-key boundary: no split */
    CHECK(sk_choose_split_kv(&p, 152, &s) == SK_OK && s == 1);
    p.max_seqlen_k = p.total_k = 42700;
    p.H = 32; /* 16 x 32 > 2 x 152: no split */
    CHECK(sk_choose_split_kv(&p, 152, &s) == SK_OK && s == 1);
    p.H = 12;

    /* a forced split: the workspace is O_part | L_part | tickets, each 256-byte aligned */
    p.split_kv = 3;
    CHECK(sk_workspace_bytes(&p, &bytes) == SK_OK);
    CHECK(bytes == a256((size_t)12 * 3 * 4096 * 128 * 4) + a256((size_t)12 * 3 * 4096 * 4) +
                       a256((size_t)1 * 12 * 16 * 4));
    /* the host-buffer call's device buffer: Q | K | V | out | LSE | workspace */
    {
        size_t ws = bytes, host = 0;
        CHECK(sk_host_buffer_bytes(&p, SK_BF16, 1, &host) == SK_OK);
        CHECK(host == a256((size_t)4096 * 12 * 192 * 2) + a256((size_t)42700 * 12 * 192 * 2) +
                          a256((size_t)42700 * 12 * 128 * 2) + a256((size_t)4096 * 12 * 128 * 2) +
                          a256((size_t)12 * 4096 * 4) + a256(ws));
    }
    p.split_kv = 1;
    CHECK(sk_workspace_bytes(&p, &bytes) == SK_OK && bytes == 0);

    /* validation before any launch */
    p.split_kv = 3;
    p.H = 0;
    CHECK(sk_workspace_bytes(&p, &bytes) == SK_ERR_INVALID_ARG);
    p.H = 12;
    p.d_qk = 96;
    p.d_v = 64;
    CHECK(sk_workspace_bytes(&p, &bytes) == SK_ERR_UNSUPPORTED);

    if (fails == 0) printf("ok\n");
    return fails == 0 ? 0 : 1;
}
