/* A plain C program using the library through include/gdn_tree.h only: no Python, no C++.
 * It exercises what needs no GPU - the version, the status strings, the workspace-size query
 * and the host-side argument checks, which return before any CUDA call - and prints "ok".
 * Built and run by tests/test_c_abi.py. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "gdn_tree.h"

static int fails = 0;
#define EXPECT(cond)                                                  \
  do {                                                                \
    if (!(cond)) {                                                    \
      fprintf(stderr, "line %d: expected %s\n", __LINE__, #cond);     \
      ++fails;                                                        \
    }                                                                 \
  } while (0)

int main(void) {
  /* any 16-byte-aligned address: the checks below fail before it would be dereferenced */
  static _Alignas(16) unsigned char dummy[64];
  const float *F = (const float *)dummy;
  float *Fo = (float *)dummy;
  const uint16_t *H = (const uint16_t *)dummy;
  const int32_t *I = (const int32_t *)dummy;
  int32_t *Io = (int32_t *)dummy;

  EXPECT(gdn_abi_version() == 3);
  EXPECT(strncmp(gdn_status_str(GDN_OK), "GDN_OK", 6) == 0);
  EXPECT(strncmp(gdn_status_str(GDN_EALIGN), "GDN_EALIGN", 10) == 0);
  EXPECT(gdn_status_str((gdn_status)99) != NULL);

  /* verify: unsupported head size, too many nodes, misaligned output, empty batch */
  EXPECT(gdn_tree_verify(F, H, H, H, F, F, I, I, 1, 1, 4, 48, 128, 4, Fo, Fo, Fo, NULL, NULL) == GDN_EINVAL);
  EXPECT(gdn_tree_verify(F, H, H, H, F, F, I, I, 1, 1, 4, 128, 128, 65, Fo, Fo, Fo, NULL, NULL) == GDN_ETOOBIG);
  EXPECT(gdn_tree_verify(F, H, H, H, F, F, I, I, 1, 1, 4, 128, 128, 4, (float *)(dummy + 4), Fo, Fo, NULL,
                         NULL) == GDN_EALIGN);
  EXPECT(gdn_tree_verify(F, H, H, H, F, F, I, I, 0, 1, 4, 128, 128, 4, Fo, Fo, Fo, NULL, NULL) == GDN_OK);

  /* commit: path array missing */
  EXPECT(gdn_tree_commit(Fo, F, F, H, I, I, NULL, I, 1, 1, 4, 128, 128, 4, NULL, NULL) == GDN_EINVAL);

  /* serving layout: 4 value heads cannot share 3 key heads */
  gdn_layout lay;
  memset(&lay, 0, sizeof lay);
  lay.H_qk = 3;
  EXPECT(gdn_tree_verify_ex(F, H, H, H, F, F, I, I, 1, 4, 4, 128, 128, 4, &lay, Fo, Fo, Fo, NULL, NULL) ==
         GDN_EINVAL);

  /* budgeting and attention argument checks */
  EXPECT(gdn_tree_budget_topb(F, 4, 0, 3, Io, NULL, NULL, NULL, NULL, NULL) == GDN_EINVAL);
  EXPECT(gdn_tree_grow_best_first(F, 4, 2, 13, 0.1f, 16, Io, Io, NULL, NULL, NULL, NULL, NULL, NULL) ==
         GDN_ETOOBIG);
  EXPECT(gdn_tree_attention(H, H, H, H, H, I, I, I, 1, 12, 4, 8, 64, 128, 4, 64, 0.1f, Fo, NULL, 0, NULL, NULL) ==
         GDN_EINVAL);
  EXPECT(gdn_tree_attention_workspace_size(0, 16, 2, 128, 8, 4096) == 0);

  if (fails) return 1;
  printf("ok\n");
  return 0;
}
