/* Uses the library from plain C99 through include/mo.h alone: the version,
 * the host-only workspace size and tile schedule, the owner planner, and the
 * argument validation that rejects calls before any CUDA work. No GPU is
 * needed; exits 0 when every check holds and prints the first failure
 * otherwise. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "mo.h"

#define CHECK(cond)                                                  \
  do {                                                               \
    if (!(cond)) {                                                   \
      fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
      return 1;                                                      \
    }                                                                \
  } while (0)

static void fake(mo_matrix* m, uintptr_t base, int64_t rows, int64_t cols) {
  const uintptr_t sz = (uintptr_t)((rows * cols * 4 + 4095) / 4096 * 4096);
  m->W = (float*)base;
  m->G = (const void*)(base + sz);
  m->V = (float*)(base + 2 * sz);
  m->rows = rows;
  m->cols = cols;
}

int main(void) {
  mo_matrix tbl[2];
  mo_muon_params p = {0.02f, 0.01f, 0.95f, 3.4445f, -4.7750f, 2.0315f, 1e-7f, 5, MO_NS_GRAM, MO_LR_ORIGINAL, 0};
  mo_tile tiles[64];
  int64_t count = -1;
  size_t ws;
  fake(&tbl[0], (uintptr_t)1 << 24, 130, 257);
  fake(&tbl[1], (uintptr_t)1 << 26, 257, 130);

  CHECK(mo_abi_version() == MO_ABI_VERSION);
  ws = mo_muon_workspace_bytes(tbl, 2, &p);
  CHECK(ws > 0);
  p.ns_steps = 0;
  CHECK(mo_muon_workspace_bytes(tbl, 2, &p) == 0);
  p.ns_steps = 5;

  /* Gram tiles of a 130 x 257 and a 257 x 130 matrix: one each (m = 130) */
  CHECK(mo_muon_tile_schedule(tbl, 2, MO_PHASE_GRAM, tiles, 64, &count) == MO_OK);
  CHECK(count == 2);
  CHECK(tiles[0].mat == 0 && tiles[1].mat == 1 && tiles[0].tm == 0 && tiles[0].tn == 0);
  /* B.X tiles: m = 130 rows by n = 257 columns is one tile row of two columns each */
  CHECK(mo_muon_tile_schedule(tbl, 2, MO_PHASE_UPDATE, tiles, 1, &count) == MO_ERR_BAD_SHAPE && count == 4);

  /* validation before any CUDA call */
  CHECK(muon_owner_step(NULL, 1, &p, (void*)((uintptr_t)1 << 30), ws, NULL) == MO_ERR_NULL_POINTER);
  CHECK(muon_owner_step(tbl, 2, &p, NULL, ws, NULL) == MO_ERR_NULL_POINTER);
  CHECK(muon_owner_step(tbl, 2, &p, (void*)(((uintptr_t)1 << 30) + 16), ws, NULL) == MO_ERR_MISALIGNED);
  CHECK(muon_owner_step(tbl, 2, &p, (void*)((uintptr_t)1 << 30), ws - 1, NULL) == MO_ERR_WORKSPACE_TOO_SMALL);
  CHECK(muon_owner_step(NULL, 0, &p, NULL, 0, NULL) == MO_OK);
  p.lr = 0.0f / 0.0f;
  CHECK(muon_owner_step(tbl, 2, &p, (void*)((uintptr_t)1 << 30), ws, NULL) == MO_ERR_BAD_PARAM);
  p.lr = 0.02f;
  tbl[1].V = tbl[0].W;
  CHECK(muon_owner_step(tbl, 2, &p, (void*)((uintptr_t)1 << 30), ws, NULL) == MO_ERR_OVERLAP);
  fake(&tbl[1], (uintptr_t)1 << 26, 257, 130);
  CHECK(mo_muon_plan_step(NULL, NULL) == MO_ERR_NULL_POINTER);
  CHECK(mo_muon_plan_lr_ptr(NULL) == NULL);
  CHECK(mo_muon_plan_destroy(NULL) == MO_OK);
  {
    mo_rmnp_params rp = {0.02f, 0.01f, 0.95f, -1.0f};
    CHECK(rmnp_step(tbl, 2, &rp, NULL) == MO_ERR_BAD_PARAM);
  }
  {
    mo_adamw_params ap = {1e-3f, 1e-2f, 0.9f, 0.95f, 1e-8f, 0};
    mo_tail_seg seg = {(float*)((uintptr_t)1 << 20), (const float*)((uintptr_t)2 << 20),
                       (float*)((uintptr_t)3 << 20), (float*)((uintptr_t)4 << 20), 1000};
    CHECK(adamw_tail_step(&seg, 1, &ap, NULL) == MO_ERR_BAD_PARAM);   /* step 0 */
  }
  CHECK(mo_status_string(MO_ERR_OVERLAP) != NULL && mo_status_string(12345) != NULL);

  /* owner planner: two roles onto two ranks */
  {
    mo_role roles[2] = {{100, 0, 0}, {50, 0, 0}};
    int32_t owner[2] = {-1, -1};
    int64_t load[2] = {0, 0};
    int32_t chosen = -1;
    CHECK(mo_plan_owners(roles, 2, 2, MO_PLAN_SCOPE_GREEDY, 0, owner, load, &chosen) == MO_OK);
    CHECK(owner[0] == 0 && owner[1] == 1 && load[0] == 100 && load[1] == 50 && chosen == MO_PLAN_SCOPE_GREEDY);
  }
  printf("ok\n");
  return 0;
}
