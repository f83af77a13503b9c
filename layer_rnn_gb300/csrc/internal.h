// Host-side declarations of every part of liblayer_rnn.so, for the API layer
// (api.cu).  Each kernel file includes only the header of its own part, so a
// change to one part's declarations does not touch the others' sources.
#pragma once

#include "gemm.h"
#include "host_common.h"
#include "rec.h"
#include "wf.h"
