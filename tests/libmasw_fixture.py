"""Locate (building if needed) the in-tree libmasw.so for the tests."""
import os

from compressed_draft_kv_gb300 import capi


def ensure_built():
    if not os.path.exists(capi.LIB_PATH):
        from compressed_draft_kv_gb300 import build
        build.build()
    return capi.load()
