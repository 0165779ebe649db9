"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/path_attn.h declares and sizes workspaces. The argument-rejection checks,
which pass fake device pointers, live in test_abi_reject.py and run only in a process
that cannot reach a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "path_attn.h")

def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(path_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("path_attn_fwd", "path_fox_fwd", "path_decode_step", "path_workspace_bytes",
              "path_status_string", "path_fwd_prepare", "path_fwd_scan", "path_check_workspace"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.library_path())
    for n in declared_functions():
        assert hasattr(so, n), n
    assert set(lib.EXPORTED) <= set(declared_functions())


def test_status_strings(lib):
    for code in range(10):
        s = lib.path_status_string(code)
        assert s.startswith("PATH_")
    assert "UNKNOWN" in lib.path_status_string(99)


def test_workspace_sizes(lib):
    # header 256 B; bf16 B1 H1 L128: qt 128*64*2, kp 2*128*64*2, dg 2*64*64*2 (fp16), and
    # the block-pair products 1*128*64*2
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 64, lib.BF16) == \
        256 + 128 * 64 * 2 + 2 * 128 * 64 * 2 + 2 * 64 * 64 * 2 + 128 * 64 * 2
    # fp32: every region fp32
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 64, lib.F32) == \
        256 + 128 * 64 * 4 + 2 * 128 * 64 * 4 + 2 * 64 * 64 * 4
    # FoX has no pair products (its scan takes one key block per step) and adds the
    # pair-relative gate sums (Lp fp32), the pair bases (hi, lo fp32 per pair), per key block
    # two fp32 bounds, one int32 extent, three fp64 block values and one fp32 key-norm
    # maximum, and per query row |q~| and the diagonal-table maximum (Lp fp32 each), each
    # region rounded up to 256 B
    fox = lib.path_workspace_bytes(lib.OP_FOX_FWD, 1, 1, 128, 64, lib.BF16)
    assert fox == lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 64, lib.BF16) - 128 * 64 * 2 + \
        512 + 8 * 256 + 2 * 512
    # ragged L rounds up to an even number of 64-token blocks
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 65, 64, lib.BF16) == \
        lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 64, lib.BF16)
    part = 4 * 2 * 66 * 4  # heads x splits x (m, l, o[64]) fp32, rounded up to 256 B
    assert lib.path_workspace_bytes(lib.OP_DECODE, 2, 2, 2048, 64, lib.BF16) == \
        256 + (part + 255) // 256 * 256
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 32, lib.BF16) == 0
    # head size 128, fp32 inputs: fp32 q~ (Lp x 128), per block [k~; P_b] (192 x 128) and
    # the fp32 diagonal table; PaTH-FoX adds the fp32 in-block and tail sums (Lp each), the
    # fp64 block totals and five per-block arrays of early-exit bounds, each rounded up to
    # 256 B
    plain = 256 + 128 * 128 * 4 + 2 * 192 * 128 * 4 + 2 * 64 * 64 * 4
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 128, lib.F32) == plain
    assert lib.path_workspace_bytes(lib.OP_FOX_FWD, 1, 1, 128, 128, lib.F32) == \
        plain + 512 + 512 + 256 + 5 * 256
    # bf16 inputs (tensor-core kernels): the same regions in bf16 with an fp16 table, the
    # block count rounded up to even; PaTH-FoX adds the fp32 in-block and tail sums (Lp
    # each), the fp64 block totals, for the early exit |q~| and the table maxima (Lp fp32
    # each) and seven per-block arrays (three fp64, three fp32, the int32 extents)
    plain16 = 256 + 128 * 128 * 2 + 2 * 192 * 128 * 2 + 2 * 64 * 64 * 2
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 128, lib.BF16) == plain16
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 65, 128, lib.BF16) == plain16
    assert lib.path_workspace_bytes(lib.OP_FOX_FWD, 1, 1, 128, 128, lib.BF16) == \
        plain16 + 512 + 512 + 256 + 512 + 512 + 7 * 256
    # decode partials (m, l, o[128])
    part128 = 4 * 2 * 130 * 4
    assert lib.path_workspace_bytes(lib.OP_DECODE, 2, 2, 2048, 128, lib.BF16) == \
        256 + (part128 + 255) // 256 * 256
    assert lib.path_workspace_bytes(lib.OP_FOX_DECODE, 2, 2, 2048, 128, lib.F32) == \
        256 + (part128 + 255) // 256 * 256
    assert lib.path_workspace_bytes(lib.OP_DECODE, 2, 2, 2048, 96, lib.BF16) == 0
    assert lib.path_workspace_bytes(lib.OP_FWD, 1, 1, 128, 64, 7) == 0
    assert lib.path_workspace_bytes(9, 1, 1, 128, 64, lib.BF16) == 0


def test_bwd_workspace_size(lib):
    # fp32 inputs: fp32 q~ (Lp x 64), [k~; P_b] (nblk x 128 x 64), diagonal logits, dq~, dk~,
    # dP_b, diagonal dT, and per pair b < a the carried query block and its logit gradient
    # (2 x 64 x 64)
    L, nb = 130, 3
    rows, blocks = nb * 64 * 64 * 4, nb * 64 * 64 * 4
    want = 256 + rows + 2 * blocks + blocks + rows + rows + blocks + blocks + 3 * 2 * 64 * 64 * 4
    assert lib.path_workspace_bytes(lib.OP_BWD, 1, 1, L, 64, lib.F32) == want
    # bf16 inputs (tensor-core query pass): the forward's bf16 preparation workspace, fp32
    # dq~, dk~ (Lp x 64), dP_b and diagonal dT (nblk x 64 x 64), and the bf16 stash: per
    # tile t of two query blocks, records b = 0 .. 2t of [X_b; dT_b] (256 x 64), i.e.
    # (blocks rounded up to even / 2)^2 records per head
    fwd = lib.path_workspace_bytes(lib.OP_FWD, 1, 1, L, 64, lib.BF16)
    npair = 2
    want16 = fwd + 2 * rows + 2 * blocks + npair * npair * 256 * 64 * 2
    assert lib.path_workspace_bytes(lib.OP_BWD, 1, 1, L, 64, lib.BF16) == want16
    fwd6 = lib.path_workspace_bytes(lib.OP_FWD, 2, 3, L, 64, lib.BF16)
    assert lib.path_workspace_bytes(lib.OP_BWD, 2, 3, L, 64, lib.BF16) == \
        fwd6 + 6 * (want16 - fwd)
    assert lib.path_workspace_bytes(lib.OP_BWD, 1, 1, 128, 96, lib.BF16) == 0


def test_bwd_d128_workspace_size(lib):
    # head size 128: the d = 128 forward's preparation workspace (fp32 for fp32 inputs, the
    # bf16 tensor-core one for bf16 inputs), then fp32 dq~, dk~ (Lp x 128), dP_b
    # (nblk x 128 x 128), diagonal dT (nblk x 64 x 64) and per pair b < a the carried query
    # block (64 x 128) and its logit gradient (64 x 64), fp32 or bf16 like the inputs;
    # PaTH-FoX adds the gate sums as at d = 64
    L, nb = 130, 3
    rows = nb * 64 * 128 * 4
    tok = nb * 64 * 4
    extra = 3 * tok + (nb * 8 + 255) // 256 * 256
    for dt, elt in ((lib.F32, 4), (lib.BF16, 2)):
        tail = 2 * rows + nb * 128 * 128 * 4 + nb * 64 * 64 * 4 + 3 * (64 * 128 + 64 * 64) * elt
        fwd = lib.path_workspace_bytes(lib.OP_FWD, 1, 1, L, 128, dt)
        assert lib.path_workspace_bytes(lib.OP_BWD, 1, 1, L, 128, dt) == fwd + tail
        fwd_fox = lib.path_workspace_bytes(lib.OP_FOX_FWD, 1, 1, L, 128, dt)
        assert lib.path_workspace_bytes(lib.OP_FOX_BWD, 1, 1, L, 128, dt) == \
            fwd_fox + tail + extra


def test_fox_bwd_workspace_size(lib):
    # the plain backward's workspace plus block-local gate sums, row and column sums of dS
    # (Lp fp32 each) and per-block fp64 gate prefixes, each region rounded up to 256 B; for
    # bf16 inputs the forward preparation part is the PaTH-FoX one
    L, nb = 130, 3
    tok = nb * 64 * 4
    extra = 3 * tok + (nb * 8 + 255) // 256 * 256
    plain = lib.path_workspace_bytes(lib.OP_BWD, 1, 1, L, 64, lib.F32)
    assert lib.path_workspace_bytes(lib.OP_FOX_BWD, 1, 1, L, 64, lib.F32) == plain + extra
    plain16 = lib.path_workspace_bytes(lib.OP_BWD, 1, 1, L, 64, lib.BF16)
    fwd = lib.path_workspace_bytes(lib.OP_FWD, 1, 1, L, 64, lib.BF16)
    fwd_fox = lib.path_workspace_bytes(lib.OP_FOX_FWD, 1, 1, L, 64, lib.BF16)
    assert lib.path_workspace_bytes(lib.OP_FOX_BWD, 1, 1, L, 64, lib.BF16) == \
        plain16 - fwd + fwd_fox + extra
    assert lib.path_workspace_bytes(lib.OP_FOX_BWD, 1, 1, L, 96, lib.BF16) == 0


@pytest.mark.gpu
def test_argument_rejection_runs_where_no_gpu_is_reachable():
    """On a machine with a GPU, the fake-pointer checks of test_abi_reject.py run in a child
    process that sees no device (CUDA_VISIBLE_DEVICES empty): a missing or misordered check
    then fails with a CUDA error instead of launching a kernel on a fake address."""
    import subprocess
    import sys
    env = dict(os.environ, CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_abi_reject.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert " passed" in r.stdout and "skipped" not in r.stdout.splitlines()[-1], r.stdout[-2000:]
