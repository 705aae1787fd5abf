"""The C ABI without a GPU: the library builds, loads, exports every symbol
include/fused_ce_tvd.h declares, and rejects bad arguments on the host
before any CUDA call (no compute is launched here)."""
import ctypes
import os
import re
import subprocess

import pytest

from distillation_ce_tvd_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fused_ce_tvd.h")

OK, INVALID, UNSUPPORTED, ALIGN = 0, 1, 2, 3
FAKE = 0x7F0000000000  # a 256-byte aligned address that is never dereferenced


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fused_ce_tvd_forward", "fused_ce_tvd_backward", "ce_forward", "ce_backward",
              "fct_status_string"):
        assert n in names
    assert set(names) == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    for n in declared_functions():
        assert n in exported, n
        assert getattr(lib, n) is not None


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version(lib):
    for code in range(5):
        assert binding.status_string(code).startswith("FCT_")
    assert "unknown" in binding.status_string(99)
    assert binding.version() >= 100


def test_no_process_wide_tuning_state(lib):
    # Tuning is a per-call argument (fct_options); nothing process-wide is
    # exported and the library reads no environment variable.
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    assert "fct_set_forward_cluster" not in out
    undefined = subprocess.run(["nm", "-D", "--undefined-only", _build.LIB_PATH],
                               capture_output=True, text=True, check=True).stdout
    assert "getenv" not in undefined
    assert binding.version() >= 400


def test_options_are_checked_per_call(lib):
    import ctypes
    base = FAKE + (3 << 30)
    args = [FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30), 0, 100, -100, base,
            base + 4096, base + 8192, base + 12288, base + 16384]

    def call(opts):
        return lib.fused_ce_tvd_forward_ex(*args, ctypes.byref(opts), None, None)
    assert call(binding.Options(0, 0, 0.0, 0)) == OK          # BT = 0, valid options
    assert call(binding.Options(3, 0, 0.0, 0)) == INVALID     # ctas_per_row
    assert call(binding.Options(16, 0, 0.0, 0)) == INVALID
    assert call(binding.Options(2, 2, 0.0, 0)) == INVALID     # l2_keep
    assert call(binding.Options(2, 0, 5.0, 0)) == INVALID     # stagger above 4
    assert call(binding.Options(2, 0, float("nan"), 0)) == INVALID
    assert call(binding.Options(2, 0, 0.0, 3)) == INVALID     # ring
    bad = binding.Options(2, 0, 0.0, 2)
    bad.reserved[3] = 1
    assert call(bad) == INVALID                               # reserved
    assert call(binding.Options(8, 1, -1.0, 2)) == OK
    assert lib.fused_ce_tvd_forward_ex(*args, None, None, None) == OK   # NULL = automatic
    fb = [FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30), 0, 100, -100,
          base, base + 256, 1, base + 512, base + 768, base + 1024, base + 1280, base + 1536,
          FAKE + (5 << 30), 128]
    assert lib.fused_ce_tvd_forward_backward_ex(*fb, ctypes.byref(binding.Options(3, 0, 0, 0)),
                                                None, None) == INVALID
    assert lib.ce_forward_backward_ex(FAKE, 128, 1, FAKE + (2 << 30), 0, 100, -100, base, 1,
                                      base + 256, base + 512, FAKE + (5 << 30), 128,
                                      ctypes.byref(binding.Options(0, 7, 0, 0)), None,
                                      None) == INVALID
    assert binding.options() is None
    assert binding.options(ctas_per_row=2).ctas_per_row == 2
    assert binding.options(ring=binding.RING_TMA).ring == 2


def test_host_entry_point_sizes_and_argument_checks(lib):
    import ctypes
    import torch
    # three slots of: two (rows, round16B(V)) logit blocks, an int64 target
    # vector, and seven fp32 vectors, each rounded up to 256 bytes; plus 256
    rup = lambda x: (x + 255) // 256 * 256  # noqa: E731
    slot = 2 * rup(4 * 104 * 2) + rup(4 * 8) + 7 * rup(4 * 4)
    assert lib.fused_ce_tvd_host_workspace_size(100, 1, 4) == 256 + 3 * slot
    slot32 = 2 * rup(5 * 12 * 4) + rup(5 * 8) + 7 * rup(5 * 4)
    assert lib.fused_ce_tvd_host_workspace_size(10, 0, 5) == 256 + 3 * slot32
    assert lib.fused_ce_tvd_host_workspace_size(0, 1, 4) == 0
    assert lib.fused_ce_tvd_host_workspace_size(100, 3, 4) == 0
    assert lib.fused_ce_tvd_host_workspace_size(100, 1, 0) == 0
    assert lib.fused_ce_tvd_host_workspace_size(100, 1, 1 << 21) == 0
    need = lib.fused_ce_tvd_host_workspace_size(100, 1, 4)
    # host buffers: real, so nothing is read unless a copy is enqueued (none is)
    s = torch.zeros(4, 100, dtype=torch.bfloat16)
    tg = torch.zeros(4, dtype=torch.int64)
    g = torch.ones(4)
    out = torch.zeros(5, 4)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    args = [P(s), 100, P(s), 100, 1, P(tg), 4, 100, -100, P(g), P(g), 1,
            P(out[0]), P(out[1]), P(out[2]), P(out[3]), P(out[4]), None, 100,
            FAKE, need, 4, None, None]
    f = lib.fused_ce_tvd_forward_backward_host

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a6=0) == OK                         # empty batch: nothing happens
    assert call(a6=-1) == INVALID
    assert call(a21=0) == INVALID                   # block_rows
    assert call(a4=9) == UNSUPPORTED
    assert call(a7=0) == INVALID                    # V
    assert call(a0=None) == INVALID
    assert call(a5=None) == INVALID
    assert call(a19=None) == INVALID                # workspace
    assert call(a1=99) == INVALID                   # ld < V
    assert call(a17=P(s), a18=50) == INVALID        # gradient ld < V
    assert call(a11=2) == INVALID                   # grad_stride
    assert call(a20=need - 1) == INVALID            # workspace one byte short
    assert call(a19=FAKE + 16) == ALIGN             # workspace not 256-byte aligned
    assert call(a5=ctypes.c_void_p(tg.data_ptr() + 4)) == ALIGN
    assert call(a21=1 << 21) == UNSUPPORTED


def fwd(lib, **kw):
    a = dict(s=FAKE, ld_s=128, t=FAKE + (1 << 30), ld_t=128, dtype=1, tg=FAKE + (2 << 30), BT=4,
             V=100, ign=-100, ce=FAKE + (3 << 30), tvd=FAKE + (3 << 30) + 4096,
             ls=FAKE + (3 << 30) + 8192, lt=FAKE + (3 << 30) + 12288,
             sg=FAKE + (3 << 30) + 16384, st=None, stream=None)
    a.update(kw)
    return lib.fused_ce_tvd_forward(a["s"], a["ld_s"], a["t"], a["ld_t"], a["dtype"], a["tg"],
                                    a["BT"], a["V"], a["ign"], a["ce"], a["tvd"], a["ls"], a["lt"],
                                    a["sg"], a["st"], a["stream"])


def bwd(lib, **kw):
    base = FAKE + (4 << 30)
    a = dict(s=FAKE, ld_s=128, t=FAKE + (1 << 30), ld_t=128, dtype=1, tg=FAKE + (2 << 30), BT=4,
             V=100, ign=-100, ls=base, lt=base + 4096, sg=base + 8192, gce=base + 12288,
             gtvd=base + 16384, gs=1, g=FAKE + (5 << 30), ld_g=128, st=None, stream=None)
    a.update(kw)
    return lib.fused_ce_tvd_backward(a["s"], a["ld_s"], a["t"], a["ld_t"], a["dtype"], a["tg"],
                                     a["BT"], a["V"], a["ign"], a["ls"], a["lt"], a["sg"], a["gce"],
                                     a["gtvd"], a["gs"], a["g"], a["ld_g"], a["st"], a["stream"])


def test_forward_argument_checks(lib):
    assert fwd(lib, BT=0) == OK
    assert fwd(lib, BT=0, s=None, t=None) == OK
    assert fwd(lib, BT=-1) == INVALID
    assert fwd(lib, V=0) == INVALID
    assert fwd(lib, dtype=7) == UNSUPPORTED
    assert fwd(lib, s=None) == INVALID
    assert fwd(lib, t=None) == INVALID
    assert fwd(lib, tg=None) == INVALID
    assert fwd(lib, sg=None) == INVALID
    assert fwd(lib, ld_s=99) == INVALID
    assert fwd(lib, ld_t=50) == INVALID
    assert fwd(lib, s=FAKE + 1) == ALIGN            # bf16 needs 2-byte alignment
    assert fwd(lib, dtype=0, s=FAKE + 2) == ALIGN   # fp32 needs 4
    assert fwd(lib, tg=FAKE + (2 << 30) + 4) == ALIGN
    assert fwd(lib, tvd=FAKE + (3 << 30)) == INVALID            # two outputs alias
    assert fwd(lib, ce=FAKE + 64) == INVALID                     # output inside the student
    assert fwd(lib, sg=FAKE + (2 << 30) + 8) == INVALID          # output inside the targets


def test_backward_argument_checks(lib):
    assert bwd(lib, BT=0) == OK
    assert bwd(lib, BT=-3) == INVALID
    assert bwd(lib, dtype=2) == UNSUPPORTED
    assert bwd(lib, gs=2) == INVALID
    assert bwd(lib, g=None) == INVALID
    assert bwd(lib, ld_g=10) == INVALID
    assert bwd(lib, g=FAKE, ld_g=256) == INVALID                  # in place needs the same ld
    assert bwd(lib, g=FAKE + 256) == INVALID                     # partial overlap with student
    assert bwd(lib, g=FAKE + (1 << 30)) == INVALID               # over the teacher
    assert bwd(lib, g=FAKE + (5 << 30) + 1) == ALIGN
    assert bwd(lib, gce=FAKE + (5 << 30) + 64) == INVALID        # grad_ce inside grad
    assert bwd(lib, lt=None) == INVALID


def test_sign_words_row_bytes_and_argument_checks(lib):
    # a uint32 tie flag, then one byte per 16-byte vector, padded to 4 bytes
    assert lib.fused_ce_tvd_signs_row_bytes(151936, 1) == 4 + 18992
    assert lib.fused_ce_tvd_signs_row_bytes(151937, 1) == 4 + 18992
    assert lib.fused_ce_tvd_signs_row_bytes(10, 0) == 4 + 4     # 2 fp32 vectors, padded
    assert lib.fused_ce_tvd_signs_row_bytes(7, 1) == 4          # no full bf16 vector
    assert lib.fused_ce_tvd_signs_row_bytes(0, 1) == 0
    assert lib.fused_ce_tvd_signs_row_bytes(100, 5) == 0
    sb = FAKE + (6 << 30)

    def fs(**kw):
        a = dict(signs=sb, ld=112, BT=4)
        a.update(kw)
        base = FAKE + (3 << 30)
        return lib.fused_ce_tvd_forward_signs(FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30),
                                              a["BT"], 100, -100, base, base + 4096, base + 8192,
                                              base + 12288, base + 16384, a["signs"], a["ld"],
                                              None, None)

    def bs(**kw):
        a = dict(signs=sb, ld=112, BT=4)
        a.update(kw)
        base = FAKE + (4 << 30)
        return lib.fused_ce_tvd_backward_signs(FAKE, 128, FAKE + (1 << 30), 128, 1,
                                               FAKE + (2 << 30), a["BT"], 100, -100, base,
                                               base + 4096, base + 8192, a["signs"], a["ld"],
                                               base + 12288, base + 16384, 1, FAKE + (5 << 30),
                                               128, None, None)

    for f in (fs, bs):
        assert f(BT=0) == OK
        assert f(signs=None) == INVALID
        assert f(ld=4 + 8) == INVALID              # V = 100 bf16 needs 4 + 12 -> 16 bytes
        assert f(ld=18) == ALIGN                    # a multiple of 4
        assert f(signs=sb + 2) == ALIGN
    assert fs(signs=FAKE + 64) == INVALID          # sign words over the student
    assert bs(signs=FAKE + (5 << 30) + 8) == INVALID  # sign words under the gradient


def test_ce_argument_checks(lib):
    assert lib.ce_forward(FAKE, 128, 1, FAKE + (2 << 30), 0, 100, -100, None, None, None, None) == OK
    assert lib.ce_forward(FAKE, 128, 1, FAKE + (2 << 30), 4, 100, -100, None,
                          FAKE + (3 << 30), None, None) == INVALID
    assert lib.ce_backward(FAKE, 128, 5, FAKE + (2 << 30), 4, 100, -100, FAKE + (3 << 30),
                           FAKE + (3 << 30) + 64, 1, FAKE + (4 << 30), 128, None, None) == UNSUPPORTED


def test_mean_argument_checks(lib):
    assert lib.fused_ce_tvd_mean_upstream(None, 4, -100, 1.0, 1.0, FAKE, FAKE + 64, None,
                                          None) == INVALID
    assert lib.fused_ce_tvd_mean_upstream(FAKE, -1, -100, 1.0, 1.0, FAKE + 256, FAKE + 512,
                                          None, None) == INVALID
    assert lib.fused_ce_tvd_mean_upstream(FAKE, 4, -100, 1.0, 1.0, FAKE + 256, FAKE + 256,
                                          None, None) == INVALID
    assert lib.fused_ce_tvd_mean_loss(FAKE, FAKE + 64, FAKE + 128, 4, -100, 1.0, 1.0, FAKE + 4,
                                      None) == INVALID          # loss inside ce
    assert lib.fused_ce_tvd_mean_loss(FAKE, FAKE + 64, FAKE + 130, 4, -100, 1.0, 1.0,
                                      FAKE + 512, None) == ALIGN


def test_forward_backward_argument_checks(lib):
    f = lib.fused_ce_tvd_forward_backward
    base = FAKE + (6 << 30)
    args = [FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30), 4, 100, -100,
            base, base + 256, 1, base + 512, base + 768, base + 1024, base + 1280, base + 1536,
            FAKE + (5 << 30), 128, None, None]
    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a6=0) == OK
    assert call(a11=3) == INVALID                  # grad_stride
    assert call(a9=None) == INVALID                # grad_ce
    assert call(a17=FAKE, a18=256) == INVALID      # in place with another ld
    assert call(a12=FAKE + (5 << 30) + 64) == INVALID   # ce inside grad
    assert call(a13=base + 512) == INVALID         # tvd aliases ce
    assert call(a17=FAKE + (5 << 30) + 1) == ALIGN       # bf16 gradient off by one byte


def test_fused_linear_workspace_sizes_and_argument_checks(lib):
    import torch
    # fp32 blocks: 2 x 4 bytes of logits + 2 x 2 of gradient (two blocks)
    # per padded entry; bf16 blocks: 3 x 2 (two student blocks, the gradient
    # over them, and the teacher's); then per row and tensor one 8-byte
    # log-sum-exp state per 256 columns
    parts = 2 * 4 * 1 * 8
    assert binding.fused_linear_ce_tvd_workspace_size(100, 4) == 4 * 104 * 12 + parts
    assert binding.fused_linear_ce_tvd_workspace_size(100, 4, torch.bfloat16) == 4 * 104 * 6 + parts
    assert binding.fused_linear_ce_tvd_workspace_size(151936, 2, torch.bfloat16) == \
        2 * 151936 * 6 + 2 * 2 * 594 * 8
    assert lib.fused_linear_ce_tvd_workspace_size(100, 4, 7) == 0
    assert lib.fused_linear_ce_tvd_workspace_size((1 << 31) - 1, (1 << 31) - 1, 1) == 0  # overflows
    assert lib.fused_linear_ce_tvd_workspace_size(0, 4, 1) == 0
    f = lib.fused_linear_ce_tvd_forward_backward
    base = FAKE + (6 << 30)
    args = [FAKE, 64, FAKE + (1 << 30), 64, 64, FAKE + (2 << 30), 64, FAKE + (3 << 30), 64, 64,
            FAKE + (4 << 30), 4, 100, -100, base, base + 256, 1,
            base + 512, base + 768, base + 1024, base + 1280, base + 1536,
            FAKE + (5 << 30), 64, FAKE + (7 << 30), 64, 1, FAKE + (8 << 30), 4 * 104 * 6 + 64, 4,
            None, None]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a26=7) == UNSUPPORTED                 # unknown logits dtype
    assert call(a28=4 * 104 * 6 + 63) == INVALID      # bf16 workspace one byte short
    assert call(a26=0) == INVALID                     # fp32 blocks need 4 * 104 * 12 + 64
    assert call(a27=FAKE + (8 << 30) + 16) == ALIGN   # workspace not 256-byte aligned
    assert call(a11=0, a26=7) == UNSUPPORTED          # the dtype is checked first
    assert call(a11=0) == OK                          # empty batch


def test_gemm_argument_checks(lib):
    assert binding.version() >= 500  # the GEMM entry point and its workspace query
    f = lib.fct_gemm_bf16
    A, B, C = FAKE, FAKE + (1 << 30), FAKE + (2 << 30)
    # A: M x K = 100 x 64 K-major (ld 64); B: N x K = 300 x 64 K-major; C: 100 x 300 fp32
    args = [A, 64, 0, B, 64, 0, C, 300, 0, 100, 300, 64, None, 0, None, None]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a8=3) == UNSUPPORTED                  # unknown output kind
    assert call(a2=2) == INVALID                      # major flag is 0 or 1
    assert call(a11=0) == INVALID                     # K >= 1
    assert call(a9=-1) == INVALID
    assert call(a9=0) == OK and call(a10=0) == OK     # empty output: nothing to do
    assert call(a0=None) == INVALID
    assert call(a1=60) == INVALID                     # lda < K
    assert call(a2=1, a1=96) == INVALID               # MN-major A needs lda >= M = 100
    assert call(a4=68) == ALIGN                       # ldb not a multiple of 8
    assert call(a0=A + 8) == ALIGN                    # A not 16-byte aligned
    assert call(a6=C + 2) == ALIGN                    # fp32 C not 4-byte aligned
    assert call(a7=299) == INVALID                    # ldc < N
    assert call(a6=A + 64) == INVALID                 # C overlaps A
    assert call(a11=1 << 31) == UNSUPPORTED           # 32-bit tile coordinates
    assert call(a9=(1 << 31) - 1000) == UNSUPPORTED   # a last tile's rows would wrap
    assert call(a13=1024) == INVALID                  # workspace bytes without a workspace
    assert call(a12=FAKE + (3 << 30) + 8, a13=1024) == ALIGN
    assert call(a12=C + 64, a13=1024) == INVALID      # workspace overlaps C
    # every split of a 300 x 1003 product: 8 parts of 512 padded rows x 1004 fp32
    assert lib.fct_gemm_bf16_workspace_size(300, 1003) == 8 * 512 * 1004 * 4
    assert lib.fct_gemm_bf16_workspace_size(0, 5) == 0
    assert lib.fct_gemm_bf16_workspace_size((1 << 31) - 1, (1 << 31) - 1) == 0  # overflows


def test_fused_linear_needs_tma_aligned_operands(lib):
    f = lib.fused_linear_ce_tvd_forward_backward
    base = FAKE + (6 << 30)
    args = [FAKE, 64, FAKE + (1 << 30), 64, 64, FAKE + (2 << 30), 64, FAKE + (3 << 30), 64, 64,
            FAKE + (4 << 30), 4, 100, -100, base, base + 256, 1,
            base + 512, base + 768, base + 1024, base + 1280, base + 1536,
            FAKE + (5 << 30), 64, FAKE + (7 << 30), 64, 1, FAKE + (8 << 30), 4 * 104 * 6 + 64, 4,
            None, None]

    def call(**kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    assert call(a1=68, a4=60) == ALIGN                # h_student row stride of 136 bytes
    assert call(a2=FAKE + (1 << 30) + 8) == ALIGN     # w_student 8 bytes off
    assert call(a7=FAKE + (3 << 30) + 2) == ALIGN     # w_teacher 2 bytes off


def test_binding_refuses_host_tensors(lib):
    import torch
    x = torch.zeros(2, 8)
    with pytest.raises(ValueError):
        binding.fused_ce_tvd_forward(x, x, torch.zeros(2, dtype=torch.int64))


def test_no_library_means_an_error_not_a_fallback(monkeypatch):
    # Without a buildable library every entry point raises: there is no CPU
    # or PyTorch path behind the binding.
    from distillation_ce_tvd_gb300 import _build

    def no_nvcc():
        raise RuntimeError("nvcc not found")

    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(_build, "_stale", lambda: True)
    monkeypatch.setattr(_build, "_nvcc", no_nvcc)
    with pytest.raises(RuntimeError):
        binding.load()
    with pytest.raises(RuntimeError):
        binding.version()


def test_plain_c_client_links_and_runs(tmp_path, lib):
    # The header and the library from C alone: compile, link, run (no GPU
    # calls; the client checks version, sizes and argument errors).
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = os.path.join(root, "distillation_ce_tvd_gb300", "libfused_ce_tvd.so")
    exe = str(tmp_path / "client")
    r = subprocess.run(["gcc", "-std=c11", "-O1", "-I", os.path.join(root, "include"),
                        os.path.join(root, "tests", "c_abi_client.c"), so,
                        "-Wl,-rpath," + os.path.dirname(so), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")


def test_vocab_shard_argument_checks(lib):
    base = FAKE + (3 << 30)
    # pass 1: (student, ld, teacher, ld, dtype, target, BT, V_shard, v_begin, ignore, part, stream)
    p1 = [FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30), 4, 100, 0, -100, base, None]

    def call(f, args, **kw):
        a = list(args)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return f(*a)
    f1 = lib.fused_ce_tvd_vp_lse
    assert call(f1, p1, a6=0) == OK
    assert call(f1, p1, a6=-1) == INVALID
    assert call(f1, p1, a8=-5) == INVALID           # v_begin
    assert call(f1, p1, a7=0) == INVALID            # V_shard
    assert call(f1, p1, a4=3) == UNSUPPORTED
    assert call(f1, p1, a10=None) == INVALID
    assert call(f1, p1, a10=base + 2) == ALIGN
    assert call(f1, p1, a10=FAKE + 64) == INVALID   # partials inside the student shard
    assert call(f1, p1, a1=99) == INVALID           # ld < V_shard
    # merge of pass 1: (parts, n_shards, target, BT, V, ignore, ce, lse_s, lse_t, status, stream)
    m1 = [base, 2, FAKE + (2 << 30), 4, 200, -100, base + 4096, base + 8192, base + 12288, None,
          None]
    fm = lib.fused_ce_tvd_vp_merge_lse
    assert call(fm, m1, a3=0) == OK
    assert call(fm, m1, a1=0) == INVALID            # no shard
    assert call(fm, m1, a4=0) == INVALID            # V
    assert call(fm, m1, a6=base + 16) == INVALID    # ce inside the partials
    assert call(fm, m1, a7=base + 4096) == INVALID  # two outputs alias
    assert call(fm, m1, a0=base + 1) == ALIGN
    # merge of pass 2: (parts, n_shards, target, BT, ignore, tvd, sigma, stream)
    m2 = [base, 3, FAKE + (2 << 30), 4, -100, base + 4096, base + 8192, None]
    ft = lib.fused_ce_tvd_vp_merge_tvd
    assert call(ft, m2, a3=0) == OK
    assert call(ft, m2, a6=None) == INVALID
    assert call(ft, m2, a6=base + 4096) == INVALID
    # backward: the shard must lie inside the vocabulary
    b4 = FAKE + (4 << 30)
    bw = [FAKE, 128, FAKE + (1 << 30), 128, 1, FAKE + (2 << 30), 4, 100, 0, 200, -100,
          b4, b4 + 4096, b4 + 8192, b4 + 12288, b4 + 16384, 1, FAKE + (5 << 30), 128, None, None]
    fb = lib.fused_ce_tvd_vp_backward
    assert call(fb, bw, a6=0) == OK
    assert call(fb, bw, a8=150) == INVALID          # v_begin + V_shard > V
    assert call(fb, bw, a9=50) == INVALID           # V < V_shard
    assert call(fb, bw, a8=-1) == INVALID
    assert call(fb, bw, a16=2) == INVALID           # grad_stride
