"""The Python binding's argument checks, run on the CPU: every buffer it hands to the library
must be on the operands' device and large enough, because the kernels would otherwise read or
write past a buffer (or through a host pointer). Tensors here are CPU tensors that report
is_cuda; the library's size queries are the real ones (host arithmetic), its compute entry
points are recorded instead of called."""
import pytest
import torch

import block_scaled_mxfp4_bf16_gb300 as mx


class _OnDevice(torch.Tensor):
    """A CPU tensor that reports is_cuda, standing for a tensor on the current CUDA device."""

    @property
    def is_cuda(self):
        return True


def dev(t: torch.Tensor) -> torch.Tensor:
    return torch.Tensor._make_subclass(_OnDevice, t)


class _Lib:
    """The real library for size queries; compute calls are recorded and succeed (a prepared
    call's creation hands out handle 1000 + its index among the calls, its runs return `run_status`)."""

    COMPUTE = ("mxfp4_quantize", "mxfp4_prepack_b", "mxfp4_gemm_ex", "mxfp4_gemm_host", "mxfp4_gemm_noalloc",
               "mxfp4_workspace_init", "mxfp4_quantize_tokens", "mxfp4_gemm_tokens", "mxfp4_call_run",
               "mxfp4_call_destroy", "mxfp4_gemm_unpacked")
    CREATE = ("mxfp4_call_create", "mxfp4_call_create_host")

    def __init__(self, real):
        self.real = real
        self.calls = []
        self.run_status = 0

    def _create(self, name, *args):
        args[-1]._obj.value = 1000 + len(self.calls)   # the handle, written through the out pointer
        self.calls.append((name, args[:-1]))
        return 0

    def __getattr__(self, name):
        if name in self.CREATE:
            return lambda *args: self._create(name, *args)
        if name == "mxfp4_call_run":
            return lambda *args: self.calls.append((name, args)) or self.run_status
        if name in self.COMPUTE:
            return lambda *args: self.calls.append((name, args)) or 0
        if name == "mxfp4_gemm_workspace_size_ex":
            return lambda *args: 0       # plans that need no workspace
        return getattr(self.real, name)


@pytest.fixture
def lib(monkeypatch):
    fake = _Lib(mx.load_library())
    monkeypatch.setattr(mx, "load_library", lambda: fake)
    monkeypatch.setattr(torch.cuda, "current_device", lambda: -1)   # a CPU tensor's get_device()
    mx._WS_NEED.clear()
    mx._PACKED_NEED.clear()
    yield fake
    mx._WS_NEED.clear()
    mx._PACKED_NEED.clear()


def _meta(*shape, dtype=torch.uint8):
    return torch.empty(*shape, dtype=dtype, device="meta")   # another device


def _gemm_operands(M=8, N=256, K=512):
    a = dev(torch.zeros(M, K, dtype=torch.bfloat16))
    packed = dev(torch.zeros(mx.mxfp4_prepack_b_size(N, K), dtype=torch.uint8))
    return a, packed, N


def test_gemm_passes_pointers_sizes_and_strides(lib):
    a, packed, N = _gemm_operands()
    c = dev(torch.zeros(8, N + 8, dtype=torch.bfloat16))[:, :N]
    mx.mxfp4_gemm(a, packed, N, c=c, stream=0)
    (name, args), = lib.calls
    assert name == "mxfp4_gemm_ex"
    assert args[:8] == (a.data_ptr(), 8, 512, 512, packed.data_ptr(), N, c.data_ptr(), N + 8)
    assert args[8] is None and args[9] == 0 and args[10] is None   # no workspace, automatic plan


def test_gemm_a_ready_sets_the_options_flag(lib):
    # a_ready is MXFP4_GEMM_A_READY in the options; alone it keeps the automatic plan (zeros)
    a, packed, N = _gemm_operands()
    mx.mxfp4_gemm(a, packed, N, stream=0, a_ready=True)
    mx.mxfp4_gemm(a, packed, N, stream=0, path=2, splits=3, a_ready=True)
    mx.prepare_gemm(a, packed, N, dev(torch.zeros(8, N, dtype=torch.bfloat16)), stream=0, a_ready=True)
    seen = [(o.path, o.splits, o.m_tile, o.flags, list(o.reserved))
            for o in (lib.calls[0][1][10]._obj, lib.calls[1][1][10]._obj, lib.calls[2][1][10]._obj)]
    assert seen == [(0, 0, 0, 1, [0] * 4), (2, 3, 0, 1, [0] * 4), (0, 0, 0, 1, [0] * 4)]
    assert lib.calls[2][0] == "mxfp4_call_create"

def test_gemm_refuses_buffers_before_any_call(lib):
    a, packed, N = _gemm_operands()
    with pytest.raises(ValueError):   # packed weights too small
        mx.mxfp4_gemm(a, packed[:1024], N, stream=0)
    with pytest.raises(ValueError):   # N past the packed tiles
        mx.mxfp4_gemm(a, packed, N + 128, stream=0)
    with pytest.raises(ValueError, match="device of the other operands"):   # on another CUDA device
        mx.mxfp4_gemm(a, dev(_meta(packed.numel())), N, stream=0)
    with pytest.raises(ValueError):   # packed weights not on a CUDA device at all
        mx.mxfp4_gemm(a, torch.zeros(packed.numel(), dtype=torch.uint8), N, stream=0)
    with pytest.raises(ValueError):   # C on another device (the kernel would store through it)
        mx.mxfp4_gemm(a, packed, N, c=_meta(8, N, dtype=torch.bfloat16), stream=0)
    with pytest.raises(ValueError):   # C of the wrong shape
        mx.mxfp4_gemm(a, packed, N, c=dev(torch.zeros(8, N - 1, dtype=torch.bfloat16)), stream=0)
    with pytest.raises(ValueError):   # workspace on another device
        mx.mxfp4_gemm(a, packed, N, workspace=_meta(1 << 20), stream=0)
    with pytest.raises(ValueError):   # workspace not contiguous
        mx.mxfp4_gemm(a, packed, N, workspace=dev(torch.zeros(64, 64, dtype=torch.uint8))[:, :32], stream=0)
    with pytest.raises(ValueError):   # K not a multiple of 8: no packed size exists
        mx.mxfp4_gemm(dev(torch.zeros(8, 100, dtype=torch.bfloat16)), packed, N, stream=0)
    with pytest.raises(ValueError):   # A on the host
        mx.mxfp4_gemm(torch.zeros(8, 512, dtype=torch.bfloat16), packed, N, stream=0)
    assert lib.calls == []


def test_gemm_refuses_a_tensor_off_the_current_device(lib, monkeypatch):
    a, packed, N = _gemm_operands()
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    with pytest.raises(ValueError):
        mx.mxfp4_gemm(a, packed, N, stream=0)
    assert lib.calls == []


def test_noalloc_checks_like_gemm(lib):
    a, packed, N = _gemm_operands()
    mx.mxfp4_gemm_noalloc(a, packed, N, stream=0)
    assert [n for n, _ in lib.calls] == ["mxfp4_gemm_noalloc"]
    with pytest.raises(ValueError):
        mx.mxfp4_gemm_noalloc(a, packed, N, c=_meta(8, N, dtype=torch.bfloat16), stream=0)
    with pytest.raises(ValueError):
        mx.mxfp4_gemm_noalloc(a, packed[:17408], N, stream=0)
    assert len(lib.calls) == 1


def test_host_call_checks(lib):
    M, N, K = 4, 256, 512
    _, packed, _ = _gemm_operands(M, N, K)
    a_host = torch.zeros(M, K, dtype=torch.bfloat16)
    c_host = torch.zeros(M, N, dtype=torch.bfloat16)
    a_dev = dev(torch.zeros(M, K, dtype=torch.bfloat16))
    c_dev = dev(torch.zeros(M, N, dtype=torch.bfloat16))
    mx.mxfp4_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, stream=0)
    (name, args), = lib.calls
    assert name == "mxfp4_gemm_host"
    assert args[:10] == (a_host.data_ptr(), M, K, K, packed.data_ptr(), N, c_host.data_ptr(), N,
                         a_dev.data_ptr(), c_dev.data_ptr())
    with pytest.raises(ValueError):   # device staging buffers must be on the device
        mx.mxfp4_gemm_host(a_host, packed, N, c_host, torch.zeros(M, K, dtype=torch.bfloat16), c_dev, stream=0)
    with pytest.raises(ValueError):   # workspace on the host
        mx.mxfp4_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, workspace=torch.zeros(64, dtype=torch.uint8),
                           stream=0)
    with pytest.raises(ValueError):   # packed weights too small
        mx.mxfp4_gemm_host(a_host, packed[:1024], N, c_host, a_dev, c_dev, stream=0)
    assert len(lib.calls) == 1


def test_quantize_checks_supplied_outputs(lib):
    rows, K = 3, 200                      # nblk = 7: the last block cut by K
    x = dev(torch.zeros(rows, K, dtype=torch.bfloat16))
    q, s = mx.mxfp4_quantize(x, stream=0)
    assert tuple(q.shape) == (rows, 7 * 16) and tuple(s.shape) == (rows, 7)
    q_ok = dev(torch.zeros(rows, 7 * 16, dtype=torch.uint8))
    s_ok = dev(torch.zeros(rows, 7, dtype=torch.uint8))
    mx.mxfp4_quantize(x, q_ok, s_ok, stream=0)
    assert [a[4:6] for _, a in lib.calls] == [(q.data_ptr(), s.data_ptr()), (q_ok.data_ptr(), s_ok.data_ptr())]
    for bad_q, bad_s in [
        (dev(torch.zeros(rows, K // 2, dtype=torch.uint8)), s_ok),        # K/2 bytes: one block short
        (q_ok, dev(torch.zeros(rows, K // 32, dtype=torch.uint8))),       # floor(K/32) scales: one short
        (_meta(rows, 7 * 16), s_ok),                                       # another device
        (q_ok, dev(torch.zeros(rows, 14, dtype=torch.uint8))[:, :7]),     # not contiguous
        (dev(torch.zeros(rows, 7 * 16, dtype=torch.int32)), s_ok),        # not bytes
    ]:
        with pytest.raises(ValueError):
            mx.mxfp4_quantize(x, bad_q, bad_s, stream=0)
    assert len(lib.calls) == 2


def test_prepack_checks(lib):
    N, K = 130, 256
    bq = dev(torch.zeros(N, K // 2, dtype=torch.uint8))
    bs = dev(torch.zeros(N, K // 32, dtype=torch.uint8))
    size = mx.mxfp4_prepack_b_size(N, K)
    out = dev(torch.zeros(size, dtype=torch.uint8))
    assert mx.mxfp4_prepack_b(bq, bs, out, stream=0) is out
    assert lib.calls[-1][1][:4] == (bq.data_ptr(), bs.data_ptr(), N, K)
    for args in [
        (bq, _meta(N, K // 32)),                                   # scales on another device
        (bq, dev(torch.zeros(N, K // 32 + 1, dtype=torch.uint8))),  # inconsistent scales
        (bq, bs, out[:-1]),                                         # packed one byte short
        (bq, bs, _meta(size)),                                      # packed on another device
        (dev(torch.zeros(N, K // 2, dtype=torch.int16)), bs),       # codes not bytes
    ]:
        with pytest.raises(ValueError):
            mx.mxfp4_prepack_b(*args, stream=0)
    assert len(lib.calls) == 1


def test_prepared_calls_pass_the_same_arguments(lib):
    # a prepared call hands the library, once, exactly what the plain call passes (without the
    # stream); each call then runs the library's handle on the stream it was prepared with, and
    # dropping the call releases the handle
    a, packed, N = _gemm_operands()
    c = dev(torch.zeros(8, N, dtype=torch.bfloat16))
    mx.mxfp4_gemm(a, packed, N, c=c, stream=0)
    call = mx.prepare_gemm(a, packed, N, c, stream=0)
    assert lib.calls[1] == ("mxfp4_call_create", lib.calls[0][1][:-1])
    call()
    call()
    assert lib.calls[2] == lib.calls[3] == ("mxfp4_call_run", (1001, 0))
    del call
    assert lib.calls[4] == ("mxfp4_call_destroy", (1001,))
    M, K = 4, 512
    _, packed, _ = _gemm_operands(M, N, K)
    a_host = torch.zeros(M, K, dtype=torch.bfloat16)
    c_host = torch.zeros(M, N, dtype=torch.bfloat16)
    a_dev = dev(torch.zeros(M, K, dtype=torch.bfloat16))
    c_dev = dev(torch.zeros(M, N, dtype=torch.bfloat16))
    mx.mxfp4_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, stream=0)
    host_call = mx.prepare_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, stream=0)
    host_call()
    assert lib.calls[5][0] == "mxfp4_gemm_host"
    assert lib.calls[6] == ("mxfp4_call_create_host", lib.calls[5][1][:-1] + (0,))
    assert lib.calls[7] == ("mxfp4_call_run", (1006, 0))
    mx.prepare_gemm_host(a_host, packed, N, c_host, a_dev, c_dev, stream=0, a_host_written=True)
    assert lib.calls[8] == ("mxfp4_call_create_host", lib.calls[5][1][:-1] + (1,))   # MXFP4_CALL_A_HOST_WRITTEN


def test_prepared_calls_check_when_prepared(lib):
    a, packed, N = _gemm_operands()
    with pytest.raises(ValueError):   # C on another device
        mx.prepare_gemm(a, packed, N, _meta(8, N, dtype=torch.bfloat16), stream=0)
    with pytest.raises(ValueError):   # packed weights too small
        mx.prepare_gemm(a, packed[:1024], N, dev(torch.zeros(8, N, dtype=torch.bfloat16)), stream=0)
    with pytest.raises(ValueError):   # host staging buffer where a device one belongs
        mx.prepare_gemm_host(torch.zeros(8, 512, dtype=torch.bfloat16), packed, N,
                             torch.zeros(8, N, dtype=torch.bfloat16), torch.zeros(8, 512, dtype=torch.bfloat16),
                             dev(torch.zeros(8, N, dtype=torch.bfloat16)), stream=0)
    assert lib.calls == []


def test_prepared_call_raises_the_library_status(lib):
    # the status word a run returns becomes the binding's exception; so does a refused creation
    a, packed, N = _gemm_operands()
    call = mx.prepare_gemm(a, packed, N, dev(torch.zeros(8, N, dtype=torch.bfloat16)), stream=0)
    call()
    lib.run_status = 4
    with pytest.raises(mx.Mxfp4Error):
        call()
    with pytest.raises(mx.Mxfp4Error):
        mx.PreparedCall(lambda *args: 2, (), 0, "mxfp4_call_create", ())


def test_token_layout_sizes():
    # the library's token tile and layout size against the layout's definition: tiles of m_tile
    # rows (cut to M rounded up to 16), 256-K steps, m_tile*128 code bytes plus two 512-byte
    # scale chunks per 128 rows
    def size(M, K, mt):
        return -(-M // mt) * -(-K // 256) * (mt * 128 + -(-mt // 128) * 1024)
    for M, K, m_tile, mt in [(64, 2048, 0, 64), (256, 7168, 0, 128), (600, 512, 0, 256), (8, 7168, 0, 16),
                             (24, 512, 0, 16), (24, 1024, 0, 32), (5, 72, 256, 16), (300, 520, 64, 64),
                             (129, 264, 256, 144), (1, 8, 0, 16)]:
        assert mx.mxfp4_token_tile(M, K, m_tile) == mt, (M, K, m_tile)
        assert mx.mxfp4_token_blocks_size(M, K, m_tile) == size(M, K, mt), (M, K, m_tile)
    for M, K, m_tile in [(0, 512, 0), (8, 100, 0), (8, 512, 24), (8, 512, 272), (8, 512, -16), (8, 0, 0)]:
        assert mx.mxfp4_token_tile(M, K, m_tile) == 0 and mx.mxfp4_token_blocks_size(M, K, m_tile) == 0


def test_token_calls_pass_pointers_and_check_buffers(lib):
    M, K, N = 40, 512, 256
    a = dev(torch.zeros(M, K + 8, dtype=torch.bfloat16))[:, :K]
    size = mx.mxfp4_token_blocks_size(M, K, 32)
    out = dev(torch.zeros(size + 256, dtype=torch.uint8))
    out = out[(-out.data_ptr()) % 256:][:size]
    tokens = mx.mxfp4_quantize_tokens(a, 32, out=out, stream=0)
    (name, args), = lib.calls
    assert name == "mxfp4_quantize_tokens"
    assert args[:7] == (a.data_ptr(), M, K, K + 8, 32, out.data_ptr(), size)
    assert tokens.data is out and (tokens.M, tokens.K, tokens.m_tile) == (M, K, 32)
    _, packed, _ = _gemm_operands(M, N, K)
    c = dev(torch.zeros(M, N + 4, dtype=torch.bfloat16))[:, :N]
    mx.mxfp4_gemm_tokens(tokens, packed, N, c=c, splits=2, stream=0)
    name, args = lib.calls[-1]
    assert name == "mxfp4_gemm_tokens"
    assert args[:10] == (out.data_ptr(), size, M, K, 32, packed.data_ptr(), N, c.data_ptr(), N + 4, 2)
    with pytest.raises(ValueError):   # output buffer one byte short
        mx.mxfp4_quantize_tokens(a, 32, out=out[:-1], stream=0)
    with pytest.raises(ValueError):   # output buffer on another device
        mx.mxfp4_quantize_tokens(a, 32, out=_meta(size), stream=0)
    with pytest.raises(ValueError):   # no layout for this token tile
        mx.mxfp4_quantize_tokens(a, 24, stream=0)
    with pytest.raises(ValueError):   # packed weights too small
        mx.mxfp4_gemm_tokens(tokens, packed[:1024], N, stream=0)
    with pytest.raises(ValueError):   # C of the wrong shape
        mx.mxfp4_gemm_tokens(tokens, packed, N, c=dev(torch.zeros(M, N - 1, dtype=torch.bfloat16)), stream=0)
    assert len(lib.calls) == 2


def test_unpacked_gemm_checks_and_arguments(lib):
    # B as the quantizer writes it: [N, ceil(K/32)*16] codes and [N, ceil(K/32)] scales; the
    # workspace handed over is 1024-byte aligned and holds B's image plus the GEMM's workspace
    M, N, K = 8, 256, 520                                  # K cuts the last 1x32 block
    nblk = -(-K // 32)
    a = dev(torch.zeros(M, K, dtype=torch.bfloat16))
    bq = dev(torch.zeros(N, nblk * 16, dtype=torch.uint8))
    bs = dev(torch.zeros(N, nblk, dtype=torch.uint8))
    need = lib.mxfp4_gemm_unpacked_workspace_size(M, N, K)   # B's image (no GEMM workspace without a GPU)
    assert need >= mx.mxfp4_prepack_b_size(N, K)
    raw = dev(torch.zeros(need + 1024, dtype=torch.uint8))
    ws = raw[(-raw.data_ptr()) % 1024:][:need]
    c = mx.mxfp4_gemm_unpacked(a, bq, bs, workspace=ws, stream=0)
    (name, args), = lib.calls
    assert name == "mxfp4_gemm_unpacked" and tuple(c.shape) == (M, N)
    assert args[:7] == (a.data_ptr(), M, K, K, bq.data_ptr(), bs.data_ptr(), N)
    assert args[9] == ws.data_ptr() and args[9] % 1024 == 0 and args[10] == need
    for bad in [
        (bq[:, :-16], bs),                                              # codes one block short
        (bq, bs[:, :-1]),                                               # scales one block short
        (_meta(N, nblk * 16), bs),                                      # codes on another device
        (dev(torch.zeros(N, nblk * 16, dtype=torch.int16)), bs),        # codes not bytes
        (bq, dev(torch.zeros(N, 2 * nblk, dtype=torch.uint8))[:, ::2]),  # scales not contiguous
    ]:
        with pytest.raises(ValueError):
            mx.mxfp4_gemm_unpacked(a, *bad, workspace=ws, stream=0)
    with pytest.raises(ValueError):   # workspace too small
        mx.mxfp4_gemm_unpacked(a, bq, bs, workspace=dev(torch.zeros(1024, dtype=torch.uint8)), stream=0)
    assert len(lib.calls) == 1
