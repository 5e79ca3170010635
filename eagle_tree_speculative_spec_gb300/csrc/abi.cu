// Library-wide entry points: status strings and version.
#include "common.cuh"

extern "C" const char *eagle3_status_string(int status) {
    switch (status) {
        case EAGLE3_OK: return "ok";
        case EAGLE3_ERR_INVALID_ARGUMENT: return "invalid argument";
        case EAGLE3_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case EAGLE3_ERR_CAPACITY: return "prefix plus tree exceeds the cache capacity";
        case EAGLE3_ERR_BAD_TREE: return "inconsistent tree parameters";
        case EAGLE3_ERR_CUDA: return "CUDA error";
        case EAGLE3_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

extern "C" int eagle3_version(void) { return 100; }
