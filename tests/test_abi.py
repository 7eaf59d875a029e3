"""The C ABI without a GPU: libpkv builds for sm_103a, loads, exports every
function include/pkv.h declares, and its structs match the binding's layout."""
import ctypes
import os
import re
import subprocess

import pytest

from paged_kv_cache_43_gb300 import build, pkv
from paged_kv_cache_43_gb300 import pool

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pkv.h")
POOL_HEADER = os.path.join(ROOT, "include", "pkv_pool.h")


def _declared_functions(header=HEADER):
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pkv.load()


def test_header_declares_the_binding_set():
    assert _declared_functions() == sorted(pkv.EXPORTED)
    assert _declared_functions(POOL_HEADER) == sorted(pool.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (pkv_\w+)", out))
    for name in _declared_functions() + _declared_functions(POOL_HEADER):
        assert name in exported, name
        assert hasattr(lib, name)


def test_status_strings(lib):
    assert pkv.status_string(0) == "ok"
    for code in range(-1, -9, -1):
        assert pkv.status_string(code) != "unknown status"
    assert pkv.status_string(-99) == "unknown status"


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "sizes.c"
    src.write_text(
        '#include <stdio.h>\n#include <stddef.h>\n#include "pkv.h"\n'
        "int main(void){printf(\"%zu %zu %zu %zu\\n\", sizeof(pkv_cache_desc),"
        " sizeof(pkv_attn_meta), offsetof(pkv_attn_meta, num_decode_seqs),"
        " offsetof(pkv_attn_meta, kv_split_tokens)); return 0;}\n")
    exe = tmp_path / "sizes"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(src), "-o",
                    str(exe)], check=True)
    got = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    assert [int(x) for x in got] == [ctypes.sizeof(pkv.CacheDesc), ctypes.sizeof(pkv.AttnMeta),
                                     pkv.AttnMeta.num_decode_seqs.offset,
                                     pkv.AttnMeta.kv_split_tokens.offset]


def test_header_compiles_as_c_and_cxx(tmp_path):
    for lang, comp in (("c", "gcc"), ("cpp", "g++")):
        src = tmp_path / f"inc.{lang}"
        src.write_text('#include "pkv.h"\n#include "pkv_pool.h"\nint main(void){return PKV_OK;}\n')
        subprocess.run([comp, "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                        str(src), "-o", str(tmp_path / f"inc_{lang}")], check=True)
