// csa_internal.h — entry points shared between the library's translation units.
// Not part of the C ABI (include/csa_index.h): no stability promise, C++ linkage.
#pragma once

#include <cstdint>

#include "csa_index.h"

// How the score-mode epilogue stores the score s of a visible record.
enum csa_fold { CSA_FOLD_MAX = 1, CSA_FOLD_ADD = 2 };

// csa_index_score with the epilogue folding each visible record's score into
// acc (same layout as the scores of csa_index_score, full mode only) instead of
// writing it: CSA_FOLD_MAX acc = max(acc, s), CSA_FOLD_ADD acc = acc + s.
// Records that are not visible (beyond the row, on an out-of-range page) leave
// acc unchanged. 128-head queries only (CSA_ERR_UNSUPPORTED otherwise); else the
// same validation and errors as csa_index_score.
csa_status csa_score_fold(const csa_index_args* args, float* acc, int64_t stride, int fold, void* stream);
