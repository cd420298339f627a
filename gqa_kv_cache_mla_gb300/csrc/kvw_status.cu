// Status strings and version of the kvw C ABI.
#include "kvw.h"

extern "C" const char* kvw_status_string(int status) {
    switch (status) {
        case KVW_OK: return "KVW_OK";
        case KVW_EINVAL: return "KVW_EINVAL: invalid argument";
        case KVW_EUNSUPPORTED: return "KVW_EUNSUPPORTED: unsupported dtype or shape";
        case KVW_ECUDA: return "KVW_ECUDA: kernel launch failed";
        default: return "unknown kvw status";
    }
}

extern "C" int kvw_version(void) { return 110; }
