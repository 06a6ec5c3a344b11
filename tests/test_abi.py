"""The C-ABI library loads and exports every entry point the header declares
(no GPU needed, no compute calls)."""

import os
import re
import subprocess

import pytest

from paged_kv_cache_attn_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in os.listdir(os.path.join(ROOT, "include")):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text,
                            flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("kv_pool_create", "kv_fork_branch", "kv_append",
                     "paged_decode_attn", "kv_free", "kv_evict"):
        assert required in names


def test_library_exports_every_declared_function():
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert hasattr(B.lib(), name)
        assert name in B.EXPORTED, f"binding lacks {name}"


def test_bytes_per_token_formula():
    # "The Reasoning Engine Meltdown", §2.1 worked example.
    assert B.kv_bytes_per_token(80, 64, 128, 2) == 2_621_440
    assert B.kv_bytes_per_token(1, 8, 128, 2) == 4096


def test_errors_carry_a_message():
    with pytest.raises(B.KVError) as e:
        B.kv_pool_create(0, 1, 1, 128)
    assert e.value.code == B.KV_ERR_INVALID_ARG
    assert "num_blocks" in str(e.value)
