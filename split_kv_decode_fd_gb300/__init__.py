"""GB300-native split-KV decode attention (Flash-Decoding).

The compute path is libfdecode.so (CUDA kernels for sm_103a behind a C ABI,
``include/fdecode.h``); this package is its thin Python binding.
"""

from .fdecode import (  # noqa: F401
    FD_AUTO_MAX_BATCH,
    FD_SPLITS_AUTO,
    FdError,
    HostDecoder,
    KvDesc,
    Workspace,
    combine,
    decode,
    decode_host,
    decode_rows,
    append_decode,
    prefill,
    attend,
    attend_backend,
    decode_static,
    static_status,
    library_path,
    load_library,
    plan_pieces,
    split_partial,
    split_size,
    workspace_bytes,
    workspace_status,
)

__version__ = "0.1.0"
