"""CPU checks of the C-ABI library: it builds, loads, exports every declared
symbol, and its host-side functions (sizes, validation, status strings) behave
as the header states.  No call here reaches the GPU."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_verification_44_gb300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_abi():
    names = declared_functions()
    assert {"spec_verify_sample", "spec_verify_greedy", "spec_verify_workspace_size",
            "spec_greedy_workspace_size", "spec_transform_probs", "spec_status_string"} <= set(names)


def test_every_declared_symbol_is_exported(lib):
    from speculative_decoding_verification_44_gb300 import _lib
    so = _lib.LIB_PATH
    for name in declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", so], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert set(declared_functions()) <= exported
    assert set(_lib.EXPORTED) == set(declared_functions())
    # nothing else leaks out of the library's namespace
    assert all(s.startswith("spec_") or s.startswith("_") for s in exported), sorted(exported)


def test_library_is_for_sm_103a(lib):
    from speculative_decoding_verification_44_gb300 import build
    cmd = build.nvcc_command()
    assert "arch=compute_103a,code=sm_103a" in " ".join(cmd)


def test_status_strings(lib):
    from speculative_decoding_verification_44_gb300 import _lib
    assert _lib.spec_status_string(0) == "ok"
    assert "workspace" in _lib.spec_status_string(4)
    assert _lib.spec_status_string(99) == "unknown status"


def test_workspace_sizes(lib):
    from speculative_decoding_verification_44_gb300 import SamplingParams, workspace_size, greedy_workspace_size
    stream = SamplingParams(0.7, 50, 0.9)
    full = SamplingParams(1.0, 0, 0.95)
    a = workspace_size(64, 5, 128256, stream, stream)
    b = workspace_size(64, 5, 128256, full, full)
    assert a > b > 0            # the kept lists only exist for the streaming top-k path
    assert a % 256 == 0 and b % 256 == 0
    assert greedy_workspace_size(256, 8) >= 256 * 4 + 256 * 9 * 8


@pytest.mark.parametrize("bad", [dict(temperature=0.0), dict(temperature=float("nan")),
                                 dict(top_p=0.0), dict(top_p=1.5), dict(top_k=-1)])
def test_invalid_params_rejected(lib, bad):
    from speculative_decoding_verification_44_gb300 import SamplingParams, _lib
    kw = dict(temperature=1.0, top_k=0, top_p=1.0)
    kw.update(bad)
    with pytest.raises(_lib.SpecError) as e:
        _lib.spec_verify_workspace_size(4, 2, 100, SamplingParams(**kw).c(), SamplingParams().c())
    assert e.value.status == _lib.SPEC_ERR_INVALID_ARG


def test_host_validation_before_any_launch(lib):
    """Arguments the contract excludes return an error and never reach the GPU."""
    from speculative_decoding_verification_44_gb300 import SamplingParams, _lib
    P = SamplingParams().c()
    fake = 1 << 20                   # 1 MiB-aligned fake device address, never dereferenced
    common = dict(d=fake, tok=fake, g=None, oh=None, ua=fake, us=fake)

    def call(tgt=fake, dtype=_lib.SPEC_BF16, B=2, G=3, V=64, ws=fake, wsb=1 << 30, out=fake):
        return _lib.spec_verify_sample(tgt, common["d"], dtype, common["tok"], None, None, common["ua"],
                                       common["us"], P, P, B, G, V, ws, wsb, out, out, None, None, None, None)

    assert call(tgt=None) == _lib.SPEC_ERR_INVALID_ARG
    assert call(dtype=7) == _lib.SPEC_ERR_INVALID_ARG
    assert call(B=0) == _lib.SPEC_ERR_INVALID_ARG
    assert call(V=0) == _lib.SPEC_ERR_INVALID_ARG
    assert call(G=-1) == _lib.SPEC_ERR_INVALID_ARG
    assert call(tgt=fake + 1) == _lib.SPEC_ERR_MISALIGNED
    assert call(ws=fake + 16) == _lib.SPEC_ERR_MISALIGNED
    assert call(wsb=16) == _lib.SPEC_ERR_WORKSPACE
    assert call(G=64) == _lib.SPEC_ERR_UNSUPPORTED        # sampling supports gamma_max <= 63
    assert _lib.spec_verify_greedy(None, 0, fake, None, 2, 3, 64, fake, 1 << 30, fake, fake, None, None) \
        == _lib.SPEC_ERR_INVALID_ARG
    assert _lib.spec_verify_greedy(fake, 0, fake, None, 2, 3, 64, fake, 8, fake, fake, None, None) \
        == _lib.SPEC_ERR_WORKSPACE
    early = _lib.spec_verify_greedy_early

    def ecall(tgt=fake, dtype=0, tok=fake, B=2, G=3, ws=fake, wsb=1 << 30, rows=None):
        return early(tgt, dtype, tok, None, B, G, 64, ws, wsb, fake, fake, None, rows, None)

    assert ecall(tgt=None) == _lib.SPEC_ERR_INVALID_ARG
    assert ecall(dtype=5) == _lib.SPEC_ERR_INVALID_ARG
    assert ecall(tok=None) == _lib.SPEC_ERR_INVALID_ARG
    assert ecall(B=0) == _lib.SPEC_ERR_INVALID_ARG
    assert ecall(ws=None) == _lib.SPEC_ERR_INVALID_ARG
    assert ecall(tgt=fake + 1) == _lib.SPEC_ERR_MISALIGNED
    assert ecall(rows=fake + 2) == _lib.SPEC_ERR_MISALIGNED
    assert ecall(ws=fake + 16) == _lib.SPEC_ERR_MISALIGNED
    assert ecall(wsb=8) == _lib.SPEC_ERR_WORKSPACE
    lenient = _lib.spec_verify_sample_lenient

    def lcall(beta, wsb=1 << 30):
        return lenient(fake, fake, 0, fake, None, None, fake, fake, P, P, beta, 2, 3, 64, fake, wsb,
                       fake, fake, None, None, None, None)

    for beta in (0.0, -1.0, 1.0000001, float("nan"), float("inf")):
        assert lcall(beta) == _lib.SPEC_ERR_INVALID_ARG, beta
    assert lcall(0.5, wsb=16) == _lib.SPEC_ERR_WORKSPACE     # a valid lenience reaches the later checks

    exf = _lib.spec_verify_sample_ex
    Pk = SamplingParams(1.0, 50, 1.0).c()

    def xcall(lenience=1.0, eos=-1, tps=None, dps=None, kept=0, tp=P, V=64, nemit=None, wsb=1 << 30):
        opt = _lib.spec_verify_options_t(lenience, eos, tps, dps, kept)
        return exf(fake, fake, 0, fake, None, None, fake, fake, tp, tp, ctypes.byref(opt), 2, 3, V, fake, wsb,
                   fake, fake, None, None, None, nemit, None)

    assert xcall(eos=64) == _lib.SPEC_ERR_INVALID_ARG                   # eos outside [-1, vocab)
    assert xcall(eos=-2) == _lib.SPEC_ERR_INVALID_ARG
    assert xcall(lenience=0.0) == _lib.SPEC_ERR_INVALID_ARG
    assert xcall(tps=fake + 2) == _lib.SPEC_ERR_MISALIGNED             # rule arrays: 4-byte aligned
    assert xcall(nemit=fake + 1) == _lib.SPEC_ERR_MISALIGNED
    assert xcall(tps=fake, kept=1) == _lib.SPEC_ERR_INVALID_ARG        # scalar rule breaks the promise
    assert xcall(tps=fake, kept=1, tp=Pk, wsb=16) == _lib.SPEC_ERR_WORKSPACE
    assert xcall(eos=5, wsb=16) == _lib.SPEC_ERR_WORKSPACE
    need = _lib.spec_verify_workspace_size_ex(2, 3, 64, Pk, Pk, _lib.spec_verify_options_t(1.0, -1, fake, fake, 0))
    kept_need = _lib.spec_verify_workspace_size_ex(2, 3, 64, Pk, Pk, _lib.spec_verify_options_t(1.0, -1, fake, fake, 1))
    plain_need = _lib.spec_verify_workspace_size(2, 3, 64, Pk, Pk)
    assert need > kept_need == plain_need                              # the promise drops the draw records

    tree = _lib.spec_verify_greedy_tree

    def tcall(tgt=fake, tok=fake, par=fake, nodes=None, N=4, ws=fake, wsb=1 << 30, path=None):
        return tree(tgt, 0, tok, par, nodes, 2, N, 64, ws, wsb, fake, fake, path, None, None)

    assert tcall(tok=None) == _lib.SPEC_ERR_INVALID_ARG
    assert tcall(par=None) == _lib.SPEC_ERR_INVALID_ARG
    assert tcall(N=0) == _lib.SPEC_ERR_INVALID_ARG
    assert tcall(par=fake + 2) == _lib.SPEC_ERR_MISALIGNED
    assert tcall(path=fake + 1) == _lib.SPEC_ERR_MISALIGNED
    assert tcall(wsb=8) == _lib.SPEC_ERR_WORKSPACE
    assert _lib.spec_tree_workspace_size(2, 4) >= 2 * 4 + 2 * 4 * 8
    assert _lib.spec_transform_probs(fake, 0, 0, 64, P, fake, None, None) == _lib.SPEC_ERR_INVALID_ARG
    assert _lib.spec_transform_probs(fake + 2, 1, 1, 64, P, fake, None, None) == _lib.SPEC_ERR_MISALIGNED


def test_product_path_has_no_oracle_dependency():
    """The package never imports the oracle (test infrastructure only)."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_44_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_struct_layouts_match_the_binding(tmp_path):
    """The ctypes mirrors of the header's structs have the C layout: a plain C
    program compiled against the header prints each struct's size and field
    offsets (gcc on the host; no GPU, no CUDA headers)."""
    import shutil
    from speculative_decoding_verification_44_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"spec_sampling_params_t": _lib.spec_sampling_params_t,
               "spec_verify_options_t": _lib.spec_verify_options_t}
    lines = ["#include <stddef.h>", "#include <stdio.h>", '#include "spec_verify.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'  printf("{name} size %zu\\n", sizeof({name}));')
        for field, _ in cls._fields_:
            lines.append(f'  printf("{name} {field} %zu\\n", offsetof({name}, {field}));')
    lines += ["  return 0;", "}"]
    src, exe = tmp_path / "layout.c", tmp_path / "layout"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = {}
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        name, field, value = line.split()
        got[(name, field)] = int(value)
    for name, cls in structs.items():
        assert got[(name, "size")] == ctypes.sizeof(cls), name
        for field, _ in cls._fields_:
            assert got[(name, field)] == getattr(cls, field).offset, (name, field)


def test_early_exit_needs_no_other_workspace(lib):
    """The early-exit stop marks and exchange words live in the leading zero region
    every sampling workspace has: the size does not depend on the option."""
    from speculative_decoding_verification_44_gb300 import _lib
    P = _lib.spec_sampling_params_t(0.7, 50, 0.9)
    sizes = []
    for early in (0, 1):
        opt = _lib.spec_verify_options_t(1.0, -1, None, None, 0, early)
        n = ctypes.c_size_t()
        assert lib.spec_verify_workspace_size_ex(64, 5, 128256, P, P, ctypes.byref(opt), ctypes.byref(n)) == 0
        sizes.append(n.value)
    plain = ctypes.c_size_t()
    assert lib.spec_verify_workspace_size(64, 5, 128256, P, P, ctypes.byref(plain)) == 0
    assert sizes[0] == sizes[1] == plain.value


def test_status_codes_match_the_binding(tmp_path):
    """The binding's status constants are the header's values (a plain C program
    compiled against the header prints them; the library asserts its kernels' codes
    against the same header at compile time)."""
    import shutil
    from speculative_decoding_verification_44_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    names = [n for n in dir(_lib) if n.startswith("SPEC_SEQ_")]
    assert "SPEC_SEQ_STALLED" in names
    lines = ["#include <stdio.h>", '#include "spec_verify.h"', "int main(void) {"]
    lines += [f'  printf("{n} %d\\n", (int){n});' for n in names]
    lines += ["  return 0;", "}"]
    src, exe = tmp_path / "codes.c", tmp_path / "codes"
    src.write_text("\n".join(lines) + "\n")
    subprocess.run([cc, "-std=c11", "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    for line in subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines():
        name, value = line.split()
        assert getattr(_lib, name) == int(value), name
