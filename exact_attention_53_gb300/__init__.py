"""GB300-native (sm_103a) exact scaled-dot-product attention forward.

The compute path is the C-ABI library ``libattn.so`` built from ``csrc/``
(declared in ``include/attn.h``); :mod:`.binding` marshals torch tensors into
it.  Importing this package loads nothing: the library is opened on first use
and a missing library raises instead of falling back to anything else.
"""

from .binding import (  # noqa: F401
    AttnError,
    attn_bwd,
    attn_bwd_general,
    attn_bwd_workspace_size,
    attn_fwd,
    attn_fwd_general,
    attn_fwd_host,
    attn_fwd_plan,
    attn_fwd_splitkv,
    attn_fwd_splitkv_noalloc,
    attn_fwd_splitkv_plan,
    attn_get_device_status,
    attn_last_error,
    bwd,
    bwd_general,
    fwd,
    fwd_general,
    fwd_splitkv_general,
    fwd_splitkv,
    library_path,
    load_library,
)
