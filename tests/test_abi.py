"""CPU-side checks of the C ABI: the shared library builds, loads and exports every
function that include/treeverify.h declares; host-side argument validation returns the
documented status codes without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "treeverify.h")


@pytest.fixture(scope="module")
def lib():
    from tree_speculative_decoding_masked_gb300 import build as b
    import tree_speculative_decoding_masked_gb300 as tv
    srcs = b.sources() + [HEADER]
    stale = (not os.path.exists(b.LIB)) or max(os.path.getmtime(s) for s in srcs) > os.path.getmtime(b.LIB)
    if stale:
        b.build()
    return tv.load_library()


def _declared():
    txt = open(HEADER).read()
    return re.findall(r"^TV_API\s+[\w\s\*]+?\b(tv_\w+)\s*\(", txt, flags=re.M)


def test_header_declares_the_boundary():
    names = set(_declared())
    for n in ("tv_tree_attention", "tv_verify_greedy", "tv_verify_sample", "tv_select_subtree", "tv_tree_prep",
              "tv_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import tree_speculative_decoding_masked_gb300 as tv
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) == set(tv.exported_symbols())


def test_status_strings(lib):
    assert lib.tv_status_string(0) == b"TV_OK"
    for code in range(-8, 0):
        assert lib.tv_status_string(code).startswith(b"TV_ERR_")
    assert lib.tv_status_string(123) == b"unknown tv_status"
    assert lib.tv_version() >> 16 == 1


NULL = None
FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first


def test_attention_host_validation(lib):
    f = lib.tv_tree_attention
    # null pointer
    assert f(NULL, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 4, 12, 0.0, 0, NULL, 0, NULL, NULL) == -1
    # Hq not a multiple of Hkv
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 6, 4, 64, 8, 4, 12, 0.0, 0, NULL, 0, NULL, NULL) == -2
    # kv stride shorter than P + N
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 4, 11, 0.0, 0, NULL, 0, NULL, NULL) == -2
    # N above the limit
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 1025, 2000, 0.0, 0, NULL, 0, NULL, NULL) == -2
    # bad dtype
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 4, 12, 0.0, 7, NULL, 0, NULL, NULL) == -3
    # negative scale
    assert f(FAKE, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 4, 12, -1.0, 0, NULL, 0, NULL, NULL) == -8
    # misaligned pointer
    odd = ctypes.c_void_p(0x1004)
    assert f(odd, FAKE, FAKE, FAKE, FAKE, 1, 4, 1, 64, 8, 4, 12, 0.0, 0, NULL, 0, NULL, NULL) == -5
    # the tensor-core path keeps split partials in cluster shared memory: no workspace
    assert lib.tv_tree_attention_workspace_size(1, 32, 8, 128, 2048, 64, 1) == 0


def test_verify_host_validation(lib):
    g = lib.tv_verify_greedy
    ws = lib.tv_verify_workspace_size(1, 16, 1024, 0, 0)
    assert ws > 0
    assert g(NULL, FAKE, FAKE, 1, 16, 1024, 0, FAKE, FAKE, FAKE, NULL, NULL, NULL, FAKE, ws, NULL, NULL) == -1
    assert g(FAKE, FAKE, FAKE, 1, 0, 1024, 0, FAKE, FAKE, FAKE, NULL, NULL, NULL, FAKE, ws, NULL, NULL) == -2
    assert g(FAKE, FAKE, FAKE, 1, 16, 1024, 0, FAKE, FAKE, FAKE, NULL, NULL, NULL, FAKE, ws - 1, NULL, NULL) == -4
    s = lib.tv_verify_sample
    wss = lib.tv_verify_workspace_size(1, 16, 1024, 0, 1)
    assert wss > ws
    assert s(FAKE, FAKE, FAKE, FAKE, 1, 16, 1024, 0.0, 1, 0, 0, FAKE, FAKE, FAKE, NULL, NULL, FAKE, wss, NULL,
             NULL) == -8
    assert s(FAKE, NULL, FAKE, FAKE, 1, 16, 1024, 1.0, 1, 0, 0, FAKE, FAKE, FAKE, NULL, NULL, FAKE, wss, NULL,
             NULL) == -1


def test_select_and_prep_host_validation(lib):
    f = lib.tv_select_subtree
    assert f(FAKE, FAKE, 1, 17, 4, 64, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL, 0, NULL, NULL) == -2
    assert f(FAKE, FAKE, 1, 16, 257, 64, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL, 0, NULL, NULL) == -2
    assert f(FAKE, FAKE, 1, 16, 4, 4097, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL, 0, NULL, NULL) == -2
    assert f(NULL, FAKE, 1, 16, 4, 64, NULL, FAKE, FAKE, FAKE, FAKE, NULL, NULL, 0, NULL, NULL) == -1
    p = lib.tv_tree_prep
    assert p(NULL, 1, 4, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL) == -1
    assert p(FAKE, 1, 2000, 0, NULL, NULL, NULL, NULL, NULL, NULL, NULL) == -2
    assert p(FAKE, 1, 4, 0, NULL, NULL, NULL, FAKE, NULL, NULL, NULL) == -1


def test_binding_has_no_cpu_fallback(monkeypatch):
    import tree_speculative_decoding_masked_gb300._binding as bnd
    monkeypatch.setattr(bnd, "_lib", None)
    monkeypatch.setattr(bnd, "_LIB_PATH", "/nonexistent/libtreeverify.so")
    with pytest.raises(RuntimeError, match="not found"):
        bnd.load_library()


def test_settings_and_utility_host_validation(lib):
    # process-wide settings: out-of-range values are refused, valid ones accepted
    assert lib.tv_set_attention_variant(6) == -8
    assert lib.tv_set_attention_variant(-1) == -8
    assert lib.tv_set_attention_splits(9) == -8
    assert lib.tv_set_sm_partition(-1, 0) == -8
    for v in (5, 4, 3, 0):
        assert lib.tv_set_attention_variant(v) == 0
    assert lib.tv_set_attention_splits(0) == 0
    # the attention plan query checks its arguments before asking the device anything
    out = ctypes.c_int(0)
    assert lib.tv_tree_attention_plan(1, 32, 8, 128, 2048, 64, 1, NULL, ctypes.byref(out)) == -1
    assert lib.tv_tree_attention_plan(1, 32, 8, 128, 2048, 64, 9, ctypes.byref(out), ctypes.byref(out)) == -3
    assert lib.tv_tree_attention_plan(1, 30, 8, 128, 2048, 64, 1, ctypes.byref(out), ctypes.byref(out)) == -2
    # Philox words: sizes, pointers, alignment
    assert lib.tv_philox4x32_10(1, FAKE, -1, FAKE, NULL) == -2
    assert lib.tv_philox4x32_10(1, NULL, 4, FAKE, NULL) == -1
    assert lib.tv_philox4x32_10(1, ctypes.c_void_p(0x1004), 4, FAKE, NULL) == -5
    # bounded-wait self-test: a status word is required and the limit is bounded
    assert lib.tv_selftest_bounded_wait(1000, NULL, NULL) == -1
    assert lib.tv_selftest_bounded_wait(0, FAKE, NULL) == -8
    assert lib.tv_selftest_bounded_wait(1000001, FAKE, NULL) == -8


class _FakeCuda:
    """Stands in for a CUDA tensor so that the binding's checks of caller-supplied
    outputs can be reached on a machine without a GPU (nothing is launched)."""

    def __init__(self, shape, dtype, device="cpu"):
        import torch
        self.shape = tuple(shape)
        self.dtype = dtype
        self.is_cuda = True
        self.device = torch.device(device)

    def is_contiguous(self):
        return True

    def numel(self):
        n = 1
        for x in self.shape:
            n *= x
        return n

    def element_size(self):
        import torch
        return torch.empty((), dtype=self.dtype).element_size()


def test_binding_refuses_host_tensors_everywhere(lib):
    # No CPU fallback: host tensors are refused as inputs, outputs, status words and
    # workspaces before anything reaches the library.
    import torch
    import tree_speculative_decoding_masked_gb300 as tv
    cpu_i32 = torch.zeros((1, 4), dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        tv.verify_greedy(torch.zeros((1, 4, 8)), cpu_i32, cpu_i32)
    with pytest.raises(ValueError, match="CUDA"):
        tv.tree_prep(cpu_i32, 0)
    with pytest.raises(ValueError, match="CUDA"):
        tv.select_subtree(torch.zeros((1, 2, 2)), torch.zeros((1, 2, 2), dtype=torch.int32), 4,
                          torch.zeros(1, dtype=torch.int32))
    logits = _FakeCuda((1, 4, 8), torch.float32)
    par, tok = _FakeCuda((1, 4), torch.int32), _FakeCuda((1, 4), torch.int32)
    outs = {"accepted_nodes": _FakeCuda((1, 4), torch.int32), "accept_len": _FakeCuda((1,), torch.int32),
            "bonus_token": _FakeCuda((1,), torch.int32), "p_draft": _FakeCuda((1, 4), torch.float32)}
    with pytest.raises(ValueError, match=r"out\['p_draft'\] must be a contiguous torch.float32"):
        tv.verify_greedy(logits, par, tok, out=dict(outs, p_draft=_FakeCuda((1, 4), torch.int32)))
    with pytest.raises(ValueError, match=r"at least 4 elements"):
        tv.verify_greedy(logits, par, tok, out=dict(outs, accepted_nodes=_FakeCuda((1, 3), torch.int32)))
    with pytest.raises(ValueError, match=r"out\['accept_len'\] must be a CUDA tensor"):
        tv.verify_greedy(logits, par, tok, out={"accept_len": torch.zeros(1, dtype=torch.int32)})
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        tv.verify_greedy(logits, par, tok, out=outs,
                         workspace=torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError, match="dev_status must be a CUDA tensor"):
        tv.verify_greedy(logits, par, tok, out=outs,
                         workspace=_FakeCuda((1 << 20,), torch.uint8), dev_status=torch.zeros(1, dtype=torch.int32))
    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        tv.frontier_topw(_FakeCuda((1, 8), torch.float32), _FakeCuda((1,), torch.int32), 2,
                         out=torch.zeros((1, 2), dtype=torch.int32))


def test_binding_refuses_inputs_the_kernels_would_misread(lib):
    # Index inputs must be int32 of exactly [B][N] (kernels read B * N entries), KV caches
    # must match the queries' batch and head size and hold P + N rows, and every tensor
    # of a call must sit on one device.  All refused before the library is called.
    import torch
    import tree_speculative_decoding_masked_gb300 as tv
    F = _FakeCuda
    logits = F((2, 4, 8), torch.float32)
    par, tok = F((2, 4), torch.int32), F((2, 4), torch.int32)
    with pytest.raises(ValueError, match="parent must be torch.int32"):
        tv.verify_greedy(logits, F((2, 4), torch.int64), tok)
    with pytest.raises(ValueError, match=r"tokens must have shape \(2, 4\)"):
        tv.verify_greedy(logits, par, F((2, 3), torch.int32))
    with pytest.raises(ValueError, match=r"parent must have shape \(2, 4\)"):
        tv.verify_greedy_static(logits, F((1, 4), torch.int32), tok)
    with pytest.raises(ValueError, match="logits must have 3 dimensions"):
        tv.verify_greedy(F((8, 8), torch.float32), par, tok)
    with pytest.raises(ValueError, match="one device per call"):
        tv.verify_greedy(F((2, 4, 8), torch.float32, "cuda:0"), F((2, 4), torch.int32, "cuda:1"),
                         F((2, 4), torch.int32, "cuda:0"))
    with pytest.raises(ValueError, match="parent must be torch.int32"):
        tv.verify_sample(logits, F((2, 4, 8), torch.float32), F((2, 4), torch.int64), tok, temperature=1.0, seed=1,
                         round=0)
    with pytest.raises(ValueError, match="dev_status must be an int32 tensor"):
        tv.verify_greedy(logits, par, tok, workspace=F((1 << 20,), torch.uint8),
                         dev_status=F((1,), torch.int64))
    q = F((2, 8, 4, 128), torch.bfloat16)
    kv = F((2, 2, 100, 128), torch.bfloat16)
    with pytest.raises(ValueError, match=r"k_cache must be \[B=2\]"):
        tv.tree_attention(q, F((1, 2, 100, 128), torch.bfloat16), F((1, 2, 100, 128), torch.bfloat16), par, 10)
    with pytest.raises(ValueError, match="prefix_len \\+ N must fit the cache rows"):
        tv.tree_attention(q, kv, kv, par, 97)
    with pytest.raises(ValueError, match="parent must be torch.int32"):
        tv.tree_attention(q, kv, kv, F((2, 4), torch.int64), 10)
    with pytest.raises(ValueError, match="one device per call"):
        tv.tree_attention(F((2, 8, 4, 128), torch.bfloat16, "cuda:0"), F((2, 2, 100, 128), torch.bfloat16, "cuda:0"),
                          F((2, 2, 100, 128), torch.bfloat16, "cuda:1"), F((2, 4), torch.int32, "cuda:0"), 10)
    with pytest.raises(ValueError, match=r"accept_len must have shape \(2,\)"):
        tv.commit_accepted_kv(kv, kv, par, F((3,), torch.int32), 10)
    with pytest.raises(ValueError, match="accepted_nodes must be torch.int32"):
        tv.commit_accepted_kv(kv, kv, F((2, 4), torch.int64), F((2,), torch.int32), 10)
    with pytest.raises(ValueError, match="root_token must have shape"):
        tv.select_subtree(F((2, 4, 4), torch.float32), F((2, 4, 4), torch.int32), 8, F((1,), torch.int32))
    with pytest.raises(ValueError, match="pool_tokens must have shape"):
        tv.select_subtree(F((2, 4, 4), torch.float32), F((2, 4, 3), torch.int32), 8, F((2,), torch.int32))
    with pytest.raises(ValueError, match="count must be torch.int32"):
        tv.frontier_topw(F((2, 16), torch.float32), F((2,), torch.int64), 4)
    with pytest.raises(ValueError, match="conf must be torch.float32"):
        tv.prune_tree(par, F((2, 4), torch.float64), 2, 4)
    with pytest.raises(ValueError, match="parent must be torch.int32"):
        tv.tree_prep(F((2, 4), torch.int16), 0)
    with pytest.raises(ValueError, match="parent_score must have shape"):
        tv.expand_children(F((3, 64), torch.float32), F((2,), torch.float32), 4)
    with pytest.raises(ValueError, match=r"counters must have shape \(5, 4\)"):
        tv.philox4x32_10(1, F((5, 3), torch.int32))


def test_header_is_plain_c_and_links_from_c(lib, tmp_path):
    # The boundary is a C ABI: the header compiles as strict C99 and a C program links
    # against the shared library and gets host-side answers from it (no GPU involved).
    import shutil
    import subprocess
    from tree_speculative_decoding_masked_gb300 import build as b
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "abi_check.c"
    src.write_text(
        '#include <stdio.h>\n#include "treeverify.h"\n'
        "int main(void) {\n"
        "  int kernel = -1, splits = -1;\n"
        '  printf("%d %d %d %d\\n", tv_version() >> 16, (int)tv_set_attention_variant(9),\n'
        "         (int)tv_tree_attention_plan(1, 4, 1, 64, 0, 16, TV_F32, NULL, &splits),\n"
        "         (int)tv_verify_workspace_size(0, 1, 1, TV_BF16, 0));\n"
        '  printf("%s\\n", tv_status_string(TV_ERR_VALUE));\n'
        "  return kernel != -1;\n}\n")
    libdir = os.path.dirname(b.LIB)
    exe = tmp_path / "abi_check"
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-l:" + os.path.basename(b.LIB),
                    "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    assert out[0].split() == ["1", str(-8), str(-1), "0"]
    assert out[1].startswith("TV_ERR_VALUE")
