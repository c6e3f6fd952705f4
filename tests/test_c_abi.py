"""The boundary as a C program sees it: include/tkg_gemm.h compiles as C99
and as C++17, a C caller links against libtkg.so (CPU), and a plain C program
(tests/c/abi_parity.c) runs each format's GEMM through the C ABI and checks it
against the oracle's C routines (GPU).  No Python or torch sits on that path."""
import os
import re
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
HEADER = os.path.join(ROOT, "include", "tkg_gemm.h")
PKG = os.path.join(ROOT, "dense_block_scaled_gb300")
ORACLE = os.path.join(ROOT, "oracle")


def _declared():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(tkg_[a-z0-9_]+)\s*\(", src)))


def _compiler(name):
    path = shutil.which(name)
    if not path:
        pytest.skip(f"{name} not available")
    return path


@pytest.mark.parametrize("lang,compiler,std", [("c", "gcc", "-std=c99"), ("c++", "g++", "-std=c++17")])
def test_header_compiles(tmp_path, lang, compiler, std):
    src = tmp_path / ("use." + ("c" if lang == "c" else "cpp"))
    refs = "\n".join(f"  (void)&{name};" for name in _declared())
    src.write_text('#include "tkg_gemm.h"\nint main(void) {\n' + refs + "\n  return 0;\n}\n")
    subprocess.run([_compiler(compiler), std, "-Wall", "-Werror", "-fsyntax-only", "-I", os.path.dirname(HEADER),
                    "-I", os.path.join(CUDA, "include"), str(src)], check=True)


def _build_c_program(out_dir):
    from dense_block_scaled_gb300 import build
    import oracle
    build.build()
    oracle.build()
    exe = os.path.join(out_dir, "abi_parity")
    subprocess.run([_compiler("gcc"), "-std=c99", "-O2", "-Wall", "-o", exe, os.path.join(ROOT, "tests", "c", "abi_parity.c"),
                    "-I", os.path.dirname(HEADER), "-I", os.path.join(CUDA, "include"),
                    "-L", PKG, "-ltkg", "-L", ORACLE, "-loracle", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
                    "-lm", f"-Wl,-rpath,{PKG}", f"-Wl,-rpath,{ORACLE}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"],
                   check=True)
    return exe


def test_c_caller_links(tmp_path):
    assert os.path.exists(_build_c_program(str(tmp_path)))


@pytest.mark.gpu
def test_c_program_parity(tmp_path):
    exe = _build_c_program(str(tmp_path))
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c abi parity: ok" in r.stdout
