/*
 * A plain C99 caller of libmok: compiles include/mok.h and include/mok_profile.h as C
 * (not C++), links the shared library, and runs the calls that need no GPU. It prints
 * one line per check ("name value") for the test that builds and runs it; exit status 0
 * means every check held.
 *
 * Checked: the status strings; the two-wave minibatch rule ("Cursor abre codigo de
 * megakernel MoE para GPUs NVL72", stamatios.com, section "Granularidade do overlap
 * computacao-comunicacao": T >= 2368 for Kimi 2.5 on 148 SMs); context creation, the
 * buffer sizes and the option setters; argument checks that return before any launch.
 */
#include <stdio.h>
#include <string.h>

#include "mok.h"
#include "mok_profile.h"

static int failures = 0;

static void expect(int cond, const char* what) {
  if (!cond) {
    printf("FAIL %s\n", what);
    ++failures;
  }
}

int main(int argc, char** argv) {
  mok_dims d;
  mok_ctx_t ctx = NULL;
  mok_sizes s;
  mok_sched sched;
  mok_status st;
  int i;
  const mok_status codes[] = {MOK_OK, MOK_ERR_INVALID_ARG, MOK_ERR_UNSUPPORTED,
                              MOK_ERR_WORKSPACE, MOK_ERR_CUDA, MOK_ERR_TIMEOUT,
                              MOK_ERR_DEVICE};
  (void)argc;
  (void)argv;

  for (i = 0; i < (int)(sizeof(codes) / sizeof(codes[0])); ++i) {
    const char* msg = mok_status_string(codes[i]);
    expect(msg != NULL && strlen(msg) > 0, "status string");
  }

  printf("minibatch_148 %d\n", mok_minibatch_tokens(7168, 2048, 8, 148));
  expect(mok_minibatch_tokens(7168, 2048, 8, 0) == -1, "minibatch rejects 0 SMs");

  memset(&d, 0, sizeof(d));
  d.T = 300;
  d.H = 256;
  d.I = 256;
  d.E = 12;
  d.k = 3;
  d.shared_I = 128;
  d.router = 1;
  st = mok_create(&d, &ctx);
  expect(st == MOK_OK && ctx != NULL, "create");
  if (ctx == NULL) return 1;
  st = mok_get_sizes(ctx, &s);
  expect(st == MOK_OK, "get_sizes");
  printf("sizes %zu %zu %zu %zu %d %d %d\n", s.aux_bytes, s.workspace_bytes, s.saved_bytes,
         s.mx_weight_bytes, s.padded_rows_max, s.macrobatches, s.ring_slots);

  expect(mok_set_precision(ctx, MOK_MXFP8) == MOK_OK, "precision mxfp8");
  expect(mok_set_precision(ctx, (mok_precision)7) == MOK_ERR_INVALID_ARG, "precision 7");
  expect(mok_set_fwd_path(ctx, MOK_FWD_LAUNCHES) == MOK_OK, "fwd path");
  expect(mok_set_wait_timeout(ctx, 1000000u) == MOK_OK, "wait timeout");
  expect(mok_set_sm_limit(ctx, -1) == MOK_ERR_INVALID_ARG, "sm limit -1");

  /* argument checks: nothing here reaches a launch */
  memset(&sched, 0, sizeof(sched));
  expect(mok_plan(ctx, NULL, NULL, NULL, &sched, NULL, NULL) == MOK_ERR_INVALID_ARG,
         "plan without a schedule");
  expect(mok_moe_fwd(ctx, &sched, NULL, NULL, NULL, NULL, NULL, NULL) == MOK_ERR_INVALID_ARG,
         "fwd without a schedule");
  expect(mok_moe_bwd(NULL, &sched, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL) ==
             MOK_ERR_INVALID_ARG,
         "bwd without a context");
  expect(mok_profile_enable(NULL, 1) == MOK_ERR_INVALID_ARG, "profile without a context");
  mok_destroy(ctx);

  d.H = 200; /* not a multiple of 128 */
  ctx = NULL;
  expect(mok_create(&d, &ctx) == MOK_ERR_INVALID_ARG && ctx == NULL, "create rejects H=200");

  printf("failures %d\n", failures);
  return failures == 0 ? 0 : 1;
}
