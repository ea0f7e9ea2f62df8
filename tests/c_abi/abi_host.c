/* Host-only use of libprism from C99: the header compiles as C, and plan
 * creation, size queries, error codes and the trace-event setter behave as
 * documented.  No device memory is touched. */
#include <stdio.h>
#include <string.h>

#include "prism.h"

#define CHECK(c)                                              \
  do {                                                        \
    if (!(c)) {                                               \
      fprintf(stderr, "check failed line %d: %s\n", __LINE__, #c); \
      return 1;                                               \
    }                                                         \
  } while (0)

static prism_config_t cfg_2k(void) {
  static const int menu[7][3] = {{1, 8, 16}, {1, 16, 8}, {2, 8, 8}, {4, 4, 8},
                                 {4, 8, 4},  {2, 4, 16}, {2, 16, 4}};
  prism_config_t c;
  memset(&c, 0, sizeof(c));
  c.B = 1; c.H = 24; c.d = 128;
  c.T = 21; c.Hg = 90; c.W = 160;
  c.zT = 3; c.zH = 16; c.zW = 16;
  c.block_tokens = 128;
  c.n_shapes = 7;
  memcpy(c.shapes, menu, sizeof(menu));
  c.Ca = 128;
  c.alpha = 1.0; c.eps = 1e-6;
  c.per_head = 1; c.use_video = 1; c.use_audio = 1;
  c.topk_floor = 8; c.topp = 0.9f;
  return c;
}

int main(void) {
  prism_config_t c = cfg_2k();
  prism_plan_t* plan = NULL;
  prism_sizes_t z;
  CHECK(prism_plan_create(&c, &plan) == PRISM_OK && plan != NULL);
  CHECK(prism_plan_query(plan, &z) == PRISM_OK);
  CHECK(z.Np == 322560 && z.Z == 420 && z.nb == 2520);
  CHECK(z.n_admissible == 2 && z.admissible[0] == 0 && z.admissible[1] == 1);
  CHECK(z.tensor_core_fwd == 1 && z.key_chunks == 3 && z.chunk_blocks == 840);
  CHECK(z.ws_bytes > 0);
  CHECK(prism_plan_set_trace_events(plan, NULL) == PRISM_OK);
  prism_plan_destroy(plan);

  /* rejections before any launch */
  c = cfg_2k(); c.d = 96 + 1;
  CHECK(prism_plan_create(&c, &plan) == PRISM_ERR_UNSUPPORTED && plan == NULL);
  c = cfg_2k(); c.shapes[0][0] = 4; c.shapes[0][1] = 16;  /* 4 x 16 x 16: 8 tiles */
  CHECK(prism_plan_create(&c, &plan) == PRISM_ERR_UNSUPPORTED);
  c = cfg_2k(); c.shapes[0][0] = 2;           /* a 256-token class that fits no 3-frame zone */
  CHECK(prism_plan_create(&c, &plan) == PRISM_ERR_NO_ADMISSIBLE_SHAPE);
  /* two block-size classes: (1,16,16) next to the 128-token menu */
  c = cfg_2k(); c.n_shapes = 8; c.shapes[7][0] = 1; c.shapes[7][1] = 16; c.shapes[7][2] = 16;
  c.class_tau[0] = 0.9;
  CHECK(prism_plan_create(&c, &plan) == PRISM_OK);
  CHECK(prism_plan_query(plan, &z) == PRISM_OK);
  CHECK(z.n_classes == 2 && z.class_tokens[0] == 128 && z.class_tokens[1] == 256);
  CHECK(z.multi_tile == 1 && z.nb == 2520 && z.blocks_per_zone == 6);
  prism_plan_destroy(plan);
  c = cfg_2k(); c.zT = 5;                     /* no menu shape divides 5 x 16 x 16 ... */
  c.n_shapes = 2; c.shapes[0][0] = 2; c.shapes[1][0] = 2;
  c.shapes[0][1] = 8; c.shapes[0][2] = 8; c.shapes[1][1] = 4; c.shapes[1][2] = 16;
  CHECK(prism_plan_create(&c, &plan) == PRISM_ERR_NO_ADMISSIBLE_SHAPE);
  c = cfg_2k(); c.key_chunk_blocks = -1;
  CHECK(prism_plan_create(&c, &plan) == PRISM_ERR_ARG);
  CHECK(prism_plan_create(NULL, &plan) == PRISM_ERR_ARG);
  CHECK(prism_plan_set_trace_events(NULL, NULL) == PRISM_ERR_ARG);
  CHECK(strcmp(prism_strerror(PRISM_ERR_DEVICE_TIMEOUT), "unknown error") != 0);
  printf("ok\n");
  return 0;
}
