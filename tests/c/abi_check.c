/* A plain C99 caller of the library: the header must compile as C and the
 * library must link and answer host-side calls without any C++ or Python in
 * between.  Exit status = number of failed checks. */
#include <stdio.h>

#include "tsv.h"

int main(void) {
  int fails = 0;
  size_t bytes = 0;
  tsv_handle h = NULL;
  tsv_status st;

  if (tsv_version() != 100) ++fails;
  if (tsv_create(NULL, 0) != TSV_ERR_INVALID_ARG) ++fails;
  if (tsv_destroy(NULL) != TSV_ERR_INVALID_ARG) ++fails;
  if (tsv_tree_verify_greedy_workspace_size(NULL, 1, 1, 10, &bytes) != TSV_ERR_INVALID_ARG) ++fails;
  if (tsv_tree_prepare(NULL, NULL, NULL, 1, NULL, NULL, NULL, NULL) != TSV_ERR_INVALID_ARG) ++fails;
  if (tsv_selftest_bounded_wait(NULL, 1, NULL, NULL, NULL) != TSV_ERR_INVALID_ARG) ++fails;

  /* Without a device: TSV_ERR_CUDA and no handle; with one: a handle to free. */
  st = tsv_create(&h, 0);
  if (st == TSV_OK) {
    if (h == NULL || tsv_destroy(h) != TSV_OK) ++fails;
  } else if (st != TSV_ERR_CUDA || h != NULL) {
    ++fails;
  }

  printf("%s | %s\n", tsv_status_string(TSV_ERR_BAD_TREE), tsv_status_string(st));
  return fails;
}
