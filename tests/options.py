"""Library options (vr_set_option) set for the duration of a block."""

import contextlib

PATH = {"auto": 0, "register": 1, "staged": 2}


@contextlib.contextmanager
def options(vr, **values):
    """Sets each named option (VR_KERNEL_PATH also takes "register" /
    "staged") and restores the previous values afterwards."""
    old = {k: vr.vr_get_option(k) for k in values}
    try:
        for k, v in values.items():
            vr.vr_set_option(k, PATH[v] if isinstance(v, str) else v)
        yield
    finally:
        for k, v in old.items():
            vr.vr_set_option(k, v)
