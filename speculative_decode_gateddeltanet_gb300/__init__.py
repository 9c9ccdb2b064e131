"""GB300 (sm_103a) GatedDeltaNet verify + commit for MTP speculative decoding.

The compute lives in ``libgdnspec.so`` (C ABI, ``include/gdnspec.h``);
``gdn`` is its ctypes binding, ``inputs`` the seeded synthetic workloads and
``build`` compiles the library in-tree.  The binding is imported lazily so
that ``inputs`` and ``build`` work before the library exists.
"""

__all__ = ["gdn", "inputs", "build"]


def __getattr__(name):
    if name in ("gdn_verify", "gdn_commit", "gdn_verify_commit", "gdn_verify_commit_static",
                "gdn_verify_deferred", "greedy_accept", "GdnArgs", "GdnPrevRows", "GdnError", "make_args",
                "make_prev", "work_bytes", "carry_bytes", "DeviceLayer", "REPLAY", "SNAPSHOT", "strerror"):
        from . import gdn

        return getattr(gdn, name)
    raise AttributeError(name)
