"""The C-ABI library loads, exports every symbol include/tfq.h declares, and
refuses bad arguments on the host before anything reaches the GPU."""
import ctypes
import os
import re

import pytest

from skinny_gemm_bit_gb300 import build as tfq_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tfq.h")


@pytest.fixture(scope="module")
def T():
    tfq_build.build()
    from skinny_gemm_bit_gb300 import tfq
    return tfq


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("tf_qlinear_pack", "tf_qlinear_run", "tf_qmlp_gateup_run", "tf_qmoe_run", "tf_decode_step_run"):
        assert n in names


def test_every_declared_symbol_is_exported(T):
    L = ctypes.CDLL(T.library_path())
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol(T):
    assert set(declared_functions()) <= set(T._SIGS)


def test_status_strings(T):
    for code, name in [(0, "TF_OK"), (1, "TF_E_INVALID_ARG"), (2, "TF_E_UNSUPPORTED_SHAPE"),
                       (3, "TF_E_WORKSPACE_TOO_SMALL"), (4, "TF_E_BAD_PACK"), (5, "TF_E_CUDA"),
                       (6, "TF_E_TIMEOUT"), (7, "TF_E_INTERNAL")]:
        assert T.status_str(code) == name
    assert T.status_str(99) == "TF_E_UNKNOWN"
    assert T.lib().tf_version() >= 10000


def test_packed_bytes(T):
    L = T.lib()
    assert L.tf_qlinear_packed_bytes(1, 3072, 1024, 4, 64) == 256 + 192 * 16 * 576
    assert L.tf_qlinear_packed_bytes(1, 3073, 1024, 4, 64) == 256 + 193 * 16 * 576   # ragged N pads to 16
    assert L.tf_qlinear_packed_bytes(128, 768, 2048, 8, 64) == 256 + 128 * 48 * 32 * 1088
    for bad in [(1, 64, 64, 3, 64), (1, 64, 64, 4, 32), (1, 64, 100, 4, 64), (1, 0, 64, 4, 64), (0, 64, 64, 4, 64),
                (1, 64, 64, 8, 16), (1, 64, 96, 4, 16)]:
        assert L.tf_qlinear_packed_bytes(*bad) == 0
    # NVFP4 (bits 4, group 16): 512 bytes of codes + 64 of block scales a 16 x 64 tile, then
    # one fp32 scale per matrix (the table padded to 16 bytes)
    assert L.tf_qlinear_packed_bytes(1, 2560, 12800, 4, 16) == 256 + 160 * 200 * 576 + 16
    assert L.tf_qlinear_packed_bytes(128, 768, 2048, 4, 16) == 256 + 128 * 48 * 32 * 576 + 512
    assert L.tf_qlinear_packed_bytes(5, 64, 64, 4, 16) == 256 + 5 * 4 * 576 + 32


FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced: validation fails first


def test_pack_refuses_bad_arguments(T):
    L = T.lib()
    d = T.tf_qweight()
    rc = L.tf_qlinear_pack(FAKE, FAKE, FAKE, 1, 64, 64, 3, 64, FAKE, 1 << 20, ctypes.byref(d), None)
    assert rc == T.TF_E_UNSUPPORTED_SHAPE and "bits" in T.last_error()
    rc = L.tf_qlinear_pack(FAKE, FAKE, FAKE, 1, 64, 96, 4, 64, FAKE, 1 << 20, ctypes.byref(d), None)
    assert rc == T.TF_E_UNSUPPORTED_SHAPE
    rc = L.tf_qlinear_pack(None, FAKE, FAKE, 1, 64, 64, 4, 64, FAKE, 1 << 20, ctypes.byref(d), None)
    assert rc == T.TF_E_INVALID_ARG
    rc = L.tf_qlinear_pack(FAKE, FAKE, FAKE, 1, 64, 64, 4, 64, ctypes.c_void_p(0x10008), 1 << 20,
                           ctypes.byref(d), None)
    assert rc == T.TF_E_INVALID_ARG and "aligned" in T.last_error()
    rc = L.tf_qlinear_pack(FAKE, FAKE, FAKE, 1, 64, 64, 4, 64, FAKE, 100, ctypes.byref(d), None)
    assert rc == T.TF_E_WORKSPACE_TOO_SMALL
    assert d.magic == 0  # nothing filled on failure


def _desc(T, N=64, K=128, bits=4, batch=1):
    d = T.tf_qweight()
    d.magic, d.version, d.bits, d.group, d.batch, d.N, d.K = 0x31515446, T.TF_PACK_VERSION, bits, 64, batch, N, K
    d.code, d.global_scale = T.TF_CODE_AFFINE, 1.0
    d.n_pad = (N + 15) // 16 * 16
    d.tile_bytes = 576 if bits == 4 else 1088
    d.matrix_bytes = d.n_pad // 16 * (K // 64) * d.tile_bytes
    d.data = 0x20000
    return d


def test_run_refuses_bad_descriptors_and_shapes(T):
    L = T.lib()
    good = _desc(T)
    ws_need = L.tf_qlinear_workspace_bytes(ctypes.byref(good), 8)
    assert ws_need >= 256

    def run(d, x=FAKE, ldx=128, M=1, y=FAKE, ydt=0, ws=FAKE, wsb=1 << 20):
        return L.tf_qlinear_run(ctypes.byref(d), x, ldx, M, None, 1e-6, None, y, ydt, ws, wsb, 0, None)

    stale = _desc(T)
    stale.magic = 0
    assert run(stale) == T.TF_E_BAD_PACK
    wrong = _desc(T)
    wrong.matrix_bytes += 16
    assert run(wrong) == T.TF_E_BAD_PACK
    assert run(_desc(T, batch=4)) == T.TF_E_UNSUPPORTED_SHAPE
    assert run(good, M=0) == T.TF_E_UNSUPPORTED_SHAPE
    assert run(good, M=9) == T.TF_E_UNSUPPORTED_SHAPE
    assert run(good, x=ctypes.c_void_p(0x10002)) == T.TF_E_INVALID_ARG
    assert run(good, ldx=100) == T.TF_E_INVALID_ARG
    assert run(good, ldx=130) == T.TF_E_INVALID_ARG
    assert run(good, ydt=7) == T.TF_E_INVALID_ARG
    assert run(good, ws=None) == T.TF_E_INVALID_ARG
    assert run(good, wsb=16) == T.TF_E_WORKSPACE_TOO_SMALL


def test_gateup_and_moe_refuse_mismatched_shapes(T):
    L = T.lib()
    g, u = _desc(T, N=64, K=128), _desc(T, N=80, K=128)
    rc = L.tf_qmlp_gateup_run(ctypes.byref(g), ctypes.byref(u), FAKE, 128, 1, None, 0.0, FAKE, FAKE, 1 << 20, 0,
                              None)
    assert rc == T.TF_E_UNSUPPORTED_SHAPE
    gate, up, down = _desc(T, 64, 128, batch=8), _desc(T, 64, 128, batch=8), _desc(T, 128, 64, batch=8)
    assert L.tf_qmoe_workspace_bytes(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), 8, 8) > 0
    bad_down = _desc(T, 128, 128, batch=8)
    assert L.tf_qmoe_workspace_bytes(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(bad_down), 8, 8) == 0
    rc = L.tf_qmoe_run(ctypes.byref(gate), ctypes.byref(up), ctypes.byref(down), FAKE, 8, 9, FAKE, FAKE, FAKE,
                       FAKE, FAKE, 1 << 30, 0, None)
    assert rc == T.TF_E_UNSUPPORTED_SHAPE


def test_tune_set_validation(T):
    assert T.lib().tf_tune_set(7, 1) == T.TF_E_INVALID_ARG
    assert T.lib().tf_tune_set(T.TF_TUNE_ROWBLOCKS, 3) == T.TF_E_INVALID_ARG
    assert T.lib().tf_tune_set(T.TF_TUNE_ROWBLOCKS, -1) == T.TF_OK


def test_workspace_query_is_independent_of_m(T):
    d = _desc(T, N=2560, K=12800)
    L = T.lib()
    sizes = {L.tf_qlinear_workspace_bytes(ctypes.byref(d), m) for m in range(1, 9)}
    assert len(sizes) == 1


def _nvfp4_desc(T, N=64, K=128):
    d = _desc(T, N, K, 4)
    d.group, d.code, d.global_scale = 16, T.TF_CODE_NVFP4, 0.004
    return d


def test_nvfp4_descriptors_are_validated(T):
    L = T.lib()
    good = _nvfp4_desc(T)
    assert L.tf_qlinear_workspace_bytes(ctypes.byref(good), 8) >= 256
    for field, value in [("group", 64), ("bits", 8), ("global_scale", float("nan")),
                         ("global_scale", float("inf")), ("code", 7)]:
        d = _nvfp4_desc(T)
        setattr(d, field, value)
        assert L.tf_qlinear_workspace_bytes(ctypes.byref(d), 8) == 0, field
    d = _desc(T)
    d.code = T.TF_CODE_NVFP4  # an affine layout (group 64) labelled NVFP4
    assert L.tf_qlinear_workspace_bytes(ctypes.byref(d), 8) == 0


def test_nvfp4_pack_refuses_bad_arguments(T):
    L = T.lib()
    d = T.tf_qweight()
    need = L.tf_qlinear_packed_bytes(1, 64, 128, 4, 16)
    assert L.tf_qlinear_pack_nvfp4(FAKE, FAKE, 1.0, 64, 100, FAKE, need, ctypes.byref(d), None) == \
        T.TF_E_UNSUPPORTED_SHAPE
    assert L.tf_qlinear_pack_nvfp4(FAKE, FAKE, float("nan"), 64, 128, FAKE, need, ctypes.byref(d), None) == \
        T.TF_E_INVALID_ARG
    assert L.tf_qlinear_pack_nvfp4(None, FAKE, 1.0, 64, 128, FAKE, need, ctypes.byref(d), None) == T.TF_E_INVALID_ARG
    assert L.tf_qlinear_pack_nvfp4(FAKE, FAKE, 1.0, 64, 128, ctypes.c_void_p(0x10008), need, ctypes.byref(d), None) == \
        T.TF_E_INVALID_ARG
    assert L.tf_qlinear_pack_nvfp4(FAKE, FAKE, 1.0, 64, 128, FAKE, need - 1, ctypes.byref(d), None) == \
        T.TF_E_WORKSPACE_TOO_SMALL
    assert d.magic == 0


def test_weight_codes_are_not_mixed(T):
    L = T.lib()
    d = _nvfp4_desc(T)
    # a stack of NVFP4 experts is a valid descriptor; a single projection of it is refused
    e2 = _nvfp4_desc(T)
    e2.batch = 2
    assert L.tf_qlinear_workspace_bytes(ctypes.byref(e2), 8) >= 256
    assert L.tf_qlinear_run(ctypes.byref(e2), FAKE, 128, 1, None, 1e-6, None, FAKE, T.TF_DTYPE_BF16, FAKE, 1 << 20, 0,
                            None) == T.TF_E_UNSUPPORTED_SHAPE
    # the MoE layer takes NVFP4 experts (gate/up [E][I][H], down [E][H][I]) ...
    g, dn = _nvfp4_desc(T, N=64, K=128), _nvfp4_desc(T, N=128, K=64)
    assert L.tf_qmoe_workspace_bytes(ctypes.byref(g), ctypes.byref(g), ctypes.byref(dn), 1, 1) > 0
    # ... but not a mix of codes
    a_dn = _desc(T, N=128, K=64)
    assert L.tf_qmoe_workspace_bytes(ctypes.byref(g), ctypes.byref(g), ctypes.byref(a_dn), 1, 1) == 0
    assert "one weight code" in T.last_error()
    # gate and up must carry the same code
    a = _desc(T)
    ws = L.tf_qmlp_gateup_run(ctypes.byref(a), ctypes.byref(d), FAKE, 128, 1, None, 1e-6, FAKE, FAKE, 1 << 20, 0,
                              None)
    assert ws == T.TF_E_UNSUPPORTED_SHAPE


def test_decoder_step_takes_one_weight_code(T):
    # a one-layer decoder (d_model 128, d_ff 128, q 64, kv 32, vocab 64): all NVFP4 is
    # planned; one affine matrix among NVFP4 ones is refused
    L = T.lib()

    def m(N, K, nv):
        return _nvfp4_desc(T, N, K) if nv else _desc(T, N, K)

    def step(nv_o):
        layer = T.tf_decoder_layer()
        layer.qkv, layer.o = m(128, 128, True), m(128, 64, nv_o)
        layer.gate, layer.up, layer.down = m(128, 128, True), m(128, 128, True), m(128, 128, True)
        layer.attn_norm = layer.mlp_norm = 0x20000
        layers = (T.tf_decoder_layer * 1)(layer)
        d = T.tf_decoder_desc()
        d.n_layers, d.d_model, d.d_ff, d.q_dim, d.kv_dim, d.vocab, d.eps = 1, 128, 128, 64, 32, 64, 1e-6
        d.layers = layers
        d.final_norm = 0x20000
        d.readout = m(64, 128, True)
        return L.tf_decode_step_workspace_bytes(ctypes.byref(d), 8)

    assert step(True) > 0
    assert step(False) == 0 and "mixes weight codes" in T.last_error()
