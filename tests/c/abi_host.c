/* A C11 caller of the library: the header compiles as C and the entry points link and answer
 * host-side argument errors (no device is needed for any call below). */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "forge.h"

static int failures = 0;

static void expect(const char *what, forge_status got, forge_status want) {
    if (got != want) {
        printf("FAIL %s: %d (%s), expected %d\n", what, (int)got, forge_status_string(got), (int)want);
        ++failures;
    }
}

int main(void) {
    forge_hparams hp;
    memset(&hp, 0, sizeof(hp));
    hp.lr = 1e-4f;
    forge_shape shape = {256, 512, 256, FORGE_STATE_FP32, 0};
    void *p = (void *)(uintptr_t)0x10000; /* aligned, never dereferenced: every call fails first */

    expect("null shape", forge_fused_dw_step(p, p, p, p, p, NULL, FORGE_ADAMW, &hp, NULL, 1, 0, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    expect("step 0", forge_fused_dw_step(p, p, p, p, p, NULL, FORGE_ADAMW, &hp, &shape, 0, 0, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    expect("misaligned W", forge_fused_dw_step(p, p, (char *)p + 8, p, p, NULL, FORGE_ADAMW, &hp, &shape, 1, 0, NULL),
           FORGE_ERR_MISALIGNED);
    forge_shape bf16_sgd = shape;
    bf16_sgd.state = FORGE_STATE_BF16;
    expect("SGD with states", forge_fused_dw_step(p, p, p, NULL, NULL, NULL, FORGE_SGD, &hp, &bf16_sgd, 1, 0, NULL),
           FORGE_ERR_UNSUPPORTED);
    expect("dX without output", forge_dx_gemm(p, p, NULL, &shape, NULL), FORGE_ERR_INVALID_ARGUMENT);
    expect("backward without dX",
           forge_linear_backward(p, p, p, p, p, NULL, NULL, FORGE_ADAMW, &hp, &shape, 1, 0, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    expect("E4M3 zero scale",
           forge_fused_dw_step_e4m3(p, p, 0.0f, 1.0f, p, p, p, NULL, FORGE_ADAMW, &hp, &shape, 1, 0, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    expect("E4M3 channel scales missing",
           forge_fused_dw_step_e4m3_channels(p, p, NULL, NULL, p, p, p, NULL, FORGE_ADAMW, &hp, &shape, 1, 0, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    forge_layer layers[2];
    memset(layers, 0, sizeof(layers));
    for (int i = 0; i < 2; ++i) {
        layers[i].dY = p; layers[i].X = p; layers[i].W = p; layers[i].m = p; layers[i].v = p;
        layers[i].T = 256; layers[i].d_out = 512; layers[i].d_in = 256; layers[i].seed = (uint64_t)i;
    }
    expect("no layers", forge_fused_dw_step_layers(NULL, 0, FORGE_STATE_FP32, FORGE_ADAMW, &hp, 1, NULL), FORGE_OK);
    expect("layers missing", forge_fused_dw_step_layers(NULL, 2, FORGE_STATE_FP32, FORGE_ADAMW, &hp, 1, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    layers[1].W = (char *)p + 8;
    expect("second layer misaligned", forge_fused_dw_step_layers(layers, 2, FORGE_STATE_FP32, FORGE_ADAMW, &hp, 1, NULL),
           FORGE_ERR_MISALIGNED);
    layers[1].W = p;
    layers[1].d_in = 100;
    expect("second layer's size", forge_fused_dw_step_layers(layers, 2, FORGE_STATE_FP32, FORGE_ADAMW, &hp, 1, NULL),
           FORGE_ERR_INVALID_ARGUMENT);
    forge_shape empty = {0, 0, 256, FORGE_STATE_FP32, 0};
    expect("empty layer", forge_fused_dw_step(NULL, NULL, NULL, NULL, NULL, NULL, FORGE_ADAMW, &hp, &empty, 1, 0, NULL),
           FORGE_OK);
    if (strcmp(forge_status_string(FORGE_ERR_TIMEOUT), "a bounded on-device wait ran out") != 0) {
        printf("FAIL status string\n");
        ++failures;
    }
    forge_set_wait_limit_ns(2000000000ull);
    (void)forge_launch_count();
    printf("%s\n", failures ? "FAILED" : "ok");
    return failures != 0;
}
