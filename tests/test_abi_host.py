"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every
symbol include/fa.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_bwd_workspace_size", "fa_status_string",
              "fa_poll_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(fa_lib):
    lib = ctypes.CDLL(fa_lib.lib_path)
    for n in _declared():
        assert hasattr(lib, n), n
    nm = subprocess.run(["nm", "-D", "--defined-only", fa_lib.lib_path], capture_output=True, text=True)
    if nm.returncode == 0:
        exported = set(re.findall(r" T (fa_[a-z0-9_]+)$", nm.stdout, flags=re.M))
        assert set(_declared()) <= exported


def test_binding_names_match_header(fa_lib):
    for n in _declared():
        assert hasattr(fa_lib, n), n


def test_status_strings(fa_lib):
    assert fa_lib.fa_status_string(fa_lib.FA_OK) == "FA_OK"
    assert fa_lib.fa_status_string(fa_lib.FA_ERR_TIMEOUT) == "FA_ERR_TIMEOUT"
    assert fa_lib.fa_status_string(99) == "FA_ERR_UNKNOWN"
    assert fa_lib.fa_version() >= 100


def test_argument_errors_before_any_cuda_call(fa_lib):
    fa = fa_lib
    p = 4096  # a 16-byte aligned fake address: never dereferenced, validation fails first
    # unsupported head size
    assert fa.fa_fwd(p, p, p, p, p, 1, 1, 64, 48, 0, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    # null pointers
    assert fa.fa_fwd(None, p, p, p, p, 1, 1, 64, 64, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    # misaligned pointer
    assert fa.fa_fwd(p + 2, p, p, p, p, 1, 1, 64, 64, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    # bad scale
    for sc in (0.0, -1.0, float("inf"), float("nan")):
        assert fa.fa_fwd(p, p, p, p, p, 1, 1, 64, 64, 0, sc, None) == fa.FA_ERR_INVALID_ARG
    # negative sizes, too many heads
    assert fa.fa_fwd(p, p, p, p, p, -1, 1, 64, 64, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_fwd(p, p, p, p, p, 1024, 1024, 64, 64, 0, 0.1, None) == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_bwd_preprocess(None, p, p, 1, 1, 8, 32, None) == fa.FA_ERR_INVALID_ARG
    # d = 32 runs the one-kernel backward, which needs the fp32 dQ workspace
    assert fa.fa_bwd(p, p, p, p, p, p, p, p, p, p, 1, 1, 64, 32, 1, 0.1, None, 0, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_bwd(p, p, p, p, p, p, p, p, p, p, 1, 1, 64, 32, 1, 0.1, p, 100, None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_debug_timeout_probe(0, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_selftest_umma(7, p, p, p, 64, 64, None) == fa.FA_ERR_INVALID_ARG


def test_empty_inputs_are_no_ops(fa_lib):
    fa = fa_lib
    assert fa.fa_fwd(None, None, None, None, None, 0, 4, 128, 64, 1, 0.125, None) == fa.FA_OK
    assert fa.fa_fwd(None, None, None, None, None, 2, 4, 0, 64, 0, 0.125, None) == fa.FA_OK
    assert fa.fa_bwd_preprocess(None, None, None, 1, 1, 0, 128, None) == fa.FA_OK
    assert fa.fa_bwd(*([None] * 10), 1, 1, 0, 128, 1, 0.1, None, 0, None) == fa.FA_OK
    assert fa.fa_bwd_workspace_size(1, 1, 0, 128, 1) == 0


def test_workspace_size(fa_lib):
    assert fa_lib.fa_bwd_workspace_size(2, 16, 4096, 128, 1) == 2 * 16 * 4096 * 128 * 4
    assert fa_lib.fa_bwd_workspace_size(1, 1, 10, 48, 0) == ctypes.c_size_t(-1).value


def test_tile_config(fa_lib):
    assert fa_lib.fa_get_tile_config(128, 0) == (0, 128, 128)
    assert fa_lib.fa_get_tile_config(128, 1) == (0, 128, 128)
    assert fa_lib.fa_get_tile_config(64, 1) == (0, 128, 128)
    assert fa_lib.fa_get_tile_config(32, 1) == (0, 128, 128)
    assert fa_lib.fa_get_tile_config(100, 0)[0] == fa_lib.FA_ERR_UNSUPPORTED
    assert fa_lib.fa_get_tile_config(128, 2)[0] == fa_lib.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("N", [1, 63, 64, 127, 128, 129, 256, 1000, 1024, 4096, 8192, 32768])
@pytest.mark.parametrize("d", [32, 64, 128])
def test_tile_pair_counts_match_closed_form(fa_lib, N, d):
    """The library's host count of tile pairs equals the oracle's closed form for
    the kernel's own tiles (the forward: query tile outer; the backward: key tile
    outer — the same set of visible pairs)."""
    for pass_ in (0, 1):
        _, br, bc = fa_lib.fa_get_tile_config(d, pass_)
        for causal in (False, True):
            assert fa_lib.fa_tile_pairs(N, d, causal, pass_) == oracle.causal_tile_pairs(N, br, bc, causal)


def test_tile_pair_counts_for_the_workloads(fa_lib):
    # 128 x 128 forward tiles: T(T+1)/2 of T^2 with the causal mask
    for N, pairs in ((1024, 36), (4096, 528), (8192, 2080), (32768, 32896)):
        assert fa_lib.fa_tile_pairs(N, 128, True, 0) == pairs
        T = N // 128
        assert fa_lib.fa_tile_pairs(N, 128, False, 0) == T * T


def test_backward_split_selection(fa_lib):
    """Form 2 (two kernels) writes dQ directly and needs no workspace; forms 1 and 3
    (one kernel, the latter persistent) need the fp32 dQ accumulator; d = 32 always
    uses form 1."""
    fa = fa_lib
    try:
        assert fa.fa_debug_set_bwd_split(4) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_debug_set_bwd_split(-1) == fa.FA_ERR_INVALID_ARG
        assert fa.fa_debug_set_bwd_split(0) == fa.FA_OK
        # d = 64 default: persistent above 3072 visible tile pairs, else two kernels
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 64, 1) == 2 * 16 * 4096 * 64 * 4  # 16896 pairs
        assert fa.fa_bwd_workspace_size(4, 8, 1024, 64, 1) == 0  # 1152 pairs
        assert fa.fa_bwd_workspace_size(4, 8, 1024, 64, 0) == 0  # 2048 pairs
        assert fa.fa_bwd_workspace_size(4, 8, 2048, 64, 1) == 4 * 8 * 2048 * 64 * 4  # 4352 pairs
        assert fa.fa_debug_set_bwd_split(2) == fa.FA_OK
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 128, 1) == 0
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 64, 1) == 0
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 32, 1) == 2 * 16 * 4096 * 32 * 4
        assert fa.fa_debug_set_bwd_split(1) == fa.FA_OK
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 128, 1) == 2 * 16 * 4096 * 128 * 4
        assert fa.fa_debug_set_bwd_split(3) == fa.FA_OK
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 128, 1) == 2 * 16 * 4096 * 128 * 4
        assert fa.fa_bwd_workspace_size(2, 16, 4096, 64, 1) == 2 * 16 * 4096 * 64 * 4
    finally:
        fa.fa_debug_set_bwd_split(0)


@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 1000), (7, 300), (128, 1000), (300, 1000), (1000, 1000), (129, 257),
                                   (8192, 8192), (32768, 32768), (4096, 8192)])
@pytest.mark.parametrize("window", [0, 1, 64, 127, 128, 129, 500, 1024])
@pytest.mark.parametrize("d", [64, 128])
def test_masked_tile_pairs_match_oracle(fa_lib, Nq, Nk, window, d):
    """The library's two-sided tile ranges give the oracle's count for every pass
    (query tiles outer and key tiles outer visit the same set of pairs)."""
    for pass_ in (0, 1):
        _, br, bc = fa_lib.fa_get_tile_config(d, pass_)
        assert fa_lib.fa_tile_pairs_ex(Nq, Nk, d, True, window, pass_) == \
            oracle.causal_tile_pairs(Nq, br, bc, True, Nk=Nk, window=window)
        if window == 0:
            assert fa_lib.fa_tile_pairs_ex(Nq, Nk, d, False, 0, pass_) == \
                oracle.causal_tile_pairs(Nq, br, bc, False, Nk=Nk)


def test_masked_argument_errors(fa_lib):
    fa = fa_lib
    p = 4096
    assert fa.fa_fwd_ex(p, p, p, p, p, 1, 1, 64, 64, 64, 0, 16, 0.1, None) == fa.FA_ERR_INVALID_ARG  # window w/o causal
    assert fa.fa_fwd_ex(p, p, p, p, p, 1, 1, 64, 64, 64, 1, -1, 0.1, None) == fa.FA_ERR_INVALID_ARG  # negative window
    assert fa.fa_fwd_ex(p, p, p, p, p, 1, 1, 65, 64, 64, 1, 0, 0.1, None) == fa.FA_ERR_UNSUPPORTED  # causal Nq > Nk
    assert fa.fa_fwd_ex(p, p, p, p, p, 1, 1, 64, 0, 64, 0, 0, 0.1, None) == fa.FA_ERR_INVALID_ARG  # no keys
    assert fa.fa_fwd_ex(None, None, None, None, None, 1, 1, 0, 64, 64, 1, 8, 0.1, None) == fa.FA_OK  # no queries
    assert fa.fa_tile_pairs_ex(65, 64, 128, 1, 0, 0) == -1
    assert fa.fa_tile_pairs_ex(64, 64, 128, 0, 8, 0) == -1
    assert fa.fa_bwd_workspace_size_ex(2, 3, 100, 700, 32, 1, 50) == 2 * 3 * 100 * 32 * 4
    assert fa.fa_bwd_workspace_size_ex(2, 3, 100, 700, 64, 1, 50) == 0  # d = 64: two kernels, no workspace
    assert fa.fa_bwd_workspace_size_ex(2, 3, 100, 700, 64, 0, 50) == ctypes.c_size_t(-1).value
    for N, c in ((1000, 0), (1000, 1), (129, 1)):
        for pass_ in (0, 1):
            assert fa.fa_tile_pairs_ex(N, N, 128, c, 0, pass_) == fa.fa_tile_pairs(N, 128, c, pass_)


def test_forward_form_switch(fa_lib):
    fa = fa_lib
    for form in (0, 1, 2, 3, 0):
        assert fa.fa_debug_set_fwd_form(form) == fa.FA_OK
    assert fa.fa_debug_set_fwd_form(4) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_set_fwd_form(-1) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("BH,Nq,Nk,d,causal,window,fwd,bwd", [
    (32, 32768, 32768, 128, 1, 0, 1, 3),   # 256 key tiles per query tile: the one-tile forward
    (32, 32768, 32768, 128, 0, 0, 1, 3),
    (32, 16384, 16384, 128, 1, 0, 3, 3),   # up to 128: persistent
    (32, 8192, 8192, 128, 1, 0, 3, 3),
    (1, 4096, 4096, 128, 0, 0, 3, 3),
    (32, 8192, 8192, 128, 1, 1024, 3, 3),  # a window: few tiles per row
    (32, 2048, 32768, 128, 1, 0, 1, 3),    # prefill: long rows; the backward is persistent at d = 128
    (32, 1024, 1024, 64, 1, 0, 3, 2),      # d = 64, 1152 tile pairs: two-kernel backward
    (128, 1024, 1024, 64, 1, 0, 3, 3),     # 4608 pairs: persistent backward
    (32, 8192, 8192, 64, 1, 0, 3, 3),
    (1, 8192, 8192, 64, 1, 0, 3, 2),       # one head, 2080 pairs
    (32, 256, 256, 32, 0, 0, 3, 1),        # d = 32: persistent forward, one-kernel backward
])
def test_selected_forms(fa_lib, BH, Nq, Nk, d, causal, window, fwd, bwd):
    assert fa_lib.fa_selected_forms(1, BH, Nq, Nk, d, causal, window) == (fa_lib.FA_OK, fwd, bwd)
    assert fa_lib.fa_selected_forms(BH, 1, Nq, Nk, d, causal, window) == (fa_lib.FA_OK, fwd, bwd)


def test_selected_forms_follow_overrides(fa_lib):
    fa = fa_lib
    try:
        fa.check(fa.fa_debug_set_fwd_form(1))
        fa.check(fa.fa_debug_set_bwd_split(2))
        assert fa.fa_selected_forms(2, 16, 4096, 4096, 128, 1, 0) == (fa.FA_OK, 1, 2)
        assert fa.fa_selected_forms(2, 16, 4096, 4096, 64, 1, 0) == (fa.FA_OK, 1, 2)
        fa.check(fa.fa_debug_set_fwd_form(2))
        assert fa.fa_selected_forms(2, 16, 4096, 4096, 64, 1, 0)[1] == 1  # two query tiles per CTA exists at d = 128 only
        fa.check(fa.fa_debug_set_bwd_split(3))
        assert fa.fa_selected_forms(1, 1, 1024, 1024, 64, 1, 0)[2] == 3
        assert fa.fa_selected_forms(1, 1, 1024, 1024, 32, 1, 0)[2] == 1  # d = 32: one kernel only
    finally:
        fa.fa_debug_set_fwd_form(0)
        fa.fa_debug_set_bwd_split(0)
    assert fa.fa_selected_forms(1, 1, 100, 100, 48, 1, 0)[0] == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_selected_forms(1, 1, 100, 100, 64, 0, 8)[0] == fa.FA_ERR_INVALID_ARG
    assert fa.fa_selected_forms(-1, 1, 100, 100, 64, 0, 0)[0] == fa.FA_ERR_INVALID_ARG


def test_bwd_plan_is_one_reading_under_a_flipping_setting(fa_lib):
    """The backward's form and its workspace size come from one reading of the form
    setting: while another thread flips fa_debug_set_bwd_split through every value,
    a form that reduces dQ in the workspace (1, 3) never comes with a zero-byte
    workspace and the two-kernel form (2) never with a non-zero one."""
    import threading

    fa = fa_lib
    B, H, N, d = 2, 3, 1000, 128
    full = B * H * N * d * 4
    stop = threading.Event()

    def flip():
        i = 0
        while not stop.is_set():
            fa.fa_debug_set_bwd_split(i % 4)
            i += 1

    t = threading.Thread(target=flip)
    t.start()
    seen = set()
    try:
        for _ in range(20000):
            st, form, need = fa.fa_debug_bwd_plan(B, H, N, N, d, True, 0)
            assert st == fa.FA_OK
            assert form in (1, 2, 3)
            assert need == (0 if form == 2 else full), (form, need)
            seen.add(form)
    finally:
        stop.set()
        t.join()
        fa.fa_debug_set_bwd_split(0)
    assert seen == {1, 2, 3}  # the flips were seen mid-loop
    assert fa.fa_debug_bwd_plan(B, H, N, N, 48, True, 0)[0] == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_debug_bwd_plan(B, H, 0, N, d, True, 0)[1:] == (3, 0)  # no query rows: nothing to reduce


def test_kernel_events_arguments(fa_lib):
    fa = fa_lib
    assert fa.fa_debug_set_kernel_events(2, None, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_set_kernel_events(0, 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_set_kernel_events(1, None, 1) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_debug_set_kernel_events(0, None, None) == fa.FA_OK
    assert fa.fa_debug_set_kernel_events(1, None, None) == fa.FA_OK
