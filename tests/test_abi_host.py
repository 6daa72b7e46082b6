"""Host-side checks of the C ABI library: it loads, exports every entry point the header
declares, and validates arguments with the pages' return codes before touching the GPU.
No GPU needed: the pointers below are never dereferenced on the host, and every case is
rejected before the first CUDA call."""
import ctypes
import os
import re

import pytest

import attention_pre_processing_gb300 as mla
from attention_pre_processing_gb300 import build as _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mla.lib()


def declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"^MLA_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, re.M)
    return names


def test_exports_every_declared_entry_point(lib):
    names = declared_functions()
    assert {"mla_prolog_workspace_size", "mla_prolog", "mla_prolog_device_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert mla.mla_prolog_status_string(0) == "MLA_OK"
    assert "161001" in mla.mla_prolog_status_string(161001)
    assert "561002" in mla.mla_prolog_status_string(561002)
    assert "561003" in mla.mla_prolog_status_string(561003)


# ---------------------------------------------------------- descriptors

BF16, I8, F32, I64 = 0, 1, 2, 3
_addr = [0x100000]


def T(dtype, *shape):
    d = mla.MlaTensor()
    _addr[0] += 0x1000
    d.data = _addr[0]
    d.dtype = dtype
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = s
    return d


def dsv3(Tk=32, **kw):
    He, Hcq, N, D, Dr, Hckv = 7168, 1536, 128, 128, 64, 512
    t = dict(x=T(BF16, Tk, He), w_dq=T(BF16, He, Hcq), w_uqqr=T(BF16, Hcq, N * (D + Dr)), w_uk=T(BF16, N, D, Hckv),
             w_dkvkr=T(BF16, He, Hckv + Dr), gamma_cq=T(BF16, Hcq), gamma_ckv=T(BF16, Hckv),
             rope_sin=T(BF16, Tk, Dr), rope_cos=T(BF16, Tk, Dr), cache_index=T(I64, Tk),
             kv_cache=T(BF16, 16, 128, 1, Hckv), kr_cache=T(BF16, 16, 128, 1, Dr),
             q_out=T(BF16, Tk, N, Hckv), q_rope_out=T(BF16, Tk, N, Dr))
    t.update(kw)
    return t


def ws_code(tensors, eps=1e-5, mode="PA_BSND"):
    try:
        mla.mla_prolog_workspace_size(tensors, eps, eps, mode)
        return 0
    except mla.MlaError as e:
        return e.code


def test_valid_arguments_pass_validation(lib):
    # Valid: validation passes and the library then asks the CUDA runtime for the device
    # (MLA_OK on a GPU machine, MLA_ERR_RUNTIME where there is no GPU).
    assert ws_code(dsv3()) in (0, 361001)
    assert ws_code(dsv3(Tk=0, x=T(BF16, 0, 7168), rope_sin=T(BF16, 0, 64), rope_cos=T(BF16, 0, 64),
                        cache_index=T(I64, 0), q_out=T(BF16, 0, 128, 512), q_rope_out=T(BF16, 0, 128, 64))) == 0


def test_null_required_tensor(lib):
    t = dsv3()
    t["w_uk"] = None
    assert ws_code(t) == 161001
    t = dsv3()
    t["x"].data = None
    assert ws_code(t) == 161001


def test_bad_shapes_and_dtypes(lib):
    assert ws_code(dsv3(w_dkvkr=T(BF16, 7168, 512))) == 161002                 # missing the rope columns
    assert ws_code(dsv3(cache_index=T(F32, 32))) == 161002                    # cacheIndex must be int64
    assert ws_code(dsv3(kv_cache=T(BF16, 16, 128, 2, 512))) == 161002         # Nkv must be 1
    assert ws_code(dsv3(q_rope_out=T(BF16, 32, 128, 32))) == 161002
    assert ws_code(dsv3(gamma_cq=T(F32, 1536))) == 161002
    assert ws_code(dsv3(), mode="PA_NZ") == 161002                            # only PA_BSND is built
    assert ws_code(dsv3(), eps=-1.0) == 161002


def test_scenario_patterns(lib):
    # int8 queryOut needs its scale output
    assert ws_code(dsv3(q_out=T(I8, 32, 128, 512))) == 161001
    assert ws_code(dsv3(q_out=T(I8, 32, 128, 512), dequant_scale_q_nope_out=T(F32, 32, 128, 1))) in (0, 361001)
    # non-quantised scenario takes no scales
    assert ws_code(dsv3(quant_scale_ckv=T(F32, 1, 512))) == 161002
    # int8 tokenX needs int8 weights and all four dequant scales
    full = dict(x=T(I8, 32, 7168), w_dq=T(I8, 7168, 1536), w_uqqr=T(I8, 1536, 24576), w_dkvkr=T(I8, 7168, 576))
    assert ws_code(dsv3(**full)) == 161001
    scales = dict(dequant_scale_x=T(F32, 32, 1), dequant_scale_w_dq=T(F32, 1, 1536),
                  dequant_scale_w_uqqr=T(F32, 1, 24576), dequant_scale_w_dkvkr=T(F32, 1, 576))
    assert ws_code(dsv3(**full, **scales)) in (0, 361001)
    assert ws_code(dsv3(**full, **scales, kv_cache=T(I8, 16, 128, 1, 512))) == 161001   # needs quantScaleCkv
    assert ws_code(dsv3(**full, **scales, kv_cache=T(I8, 16, 128, 1, 512),
                        quant_scale_ckv=T(F32, 1, 512))) in (0, 361001)
    # partial quantisation with int8 caches needs both cache scales
    part = dict(w_uqqr=T(I8, 1536, 24576), dequant_scale_w_uqqr=T(F32, 1, 24576))
    assert ws_code(dsv3(**part)) in (0, 361001)
    assert ws_code(dsv3(**part, kv_cache=T(I8, 16, 128, 1, 512), quant_scale_ckv=T(F32, 1, 512))) == 161002
    assert ws_code(dsv3(**part, kv_cache=T(I8, 16, 128, 1, 512), kr_cache=T(I8, 16, 128, 1, 64),
                        quant_scale_ckv=T(F32, 1, 512), quant_scale_ckr=T(F32, 1, 64))) in (0, 361001)


def test_tiling_rules(lib):
    He = 7168
    t = dsv3(w_dq=T(BF16, He, 1500), w_uqqr=T(BF16, 1500, 24576), gamma_cq=T(BF16, 1500))
    assert ws_code(t) == 561002                                               # Hcq % 64
    t = dsv3(q_out=T(I8, 32, 128, 1024), dequant_scale_q_nope_out=T(F32, 32, 128, 1),
             w_uk=T(BF16, 128, 128, 1024), w_dkvkr=T(BF16, He, 1024 + 64), gamma_ckv=T(BF16, 1024),
             kv_cache=T(BF16, 16, 128, 1, 1024))
    assert ws_code(t) == 561002                                               # int8 row longer than 512


def test_misaligned_pointer(lib):
    t = dsv3()
    t["x"].data = t["x"].data + 2
    assert ws_code(t) == 161002


def test_batch_seq_views_accepted(lib):
    t = dsv3(x=T(BF16, 4, 8, 7168), rope_sin=T(BF16, 4, 8, 64), rope_cos=T(BF16, 4, 8, 64),
             cache_index=T(I64, 4, 8), q_out=T(BF16, 4, 8, 128, 512), q_rope_out=T(BF16, 4, 8, 128, 64))
    assert ws_code(t) in (0, 361001)


def test_product_has_no_cpu_fallback():
    """The package never reaches for the oracle: no module of it imports or names it."""
    pkg = os.path.join(ROOT, "attention_pre_processing_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text and "mla_oracle" not in text, fn


# ---------------------------------------------------------- the aclnnMlaPreprocess variant

F16, I32 = 4, 5


def pp(Tk=32, dt=BF16, mode=0, **kw):
    He, Hcq, N, D = 7168, 1536, 128, 128
    n1, n2 = Hcq + 576, N * (D + 64)
    kv = T(dt, 192, 128, 1, 576 if mode == 0 else 512)
    t = dict(input=T(dt, Tk, He), gamma0=T(dt, He), beta0=T(dt, He), quant_scale0=T(dt, 1), quant_offset0=T(I8, 1),
             wdqkv=T(I8, n1, He), de_scale0=T(F32, n1), bias0=T(I32, n1), gamma1=T(dt, Hcq), beta1=T(dt, Hcq),
             quant_scale1=T(dt, 1), quant_offset1=T(I8, 1), wuq=T(I8, n2, Hcq), de_scale1=T(F32, n2),
             bias1=T(I32, n2), gamma2=T(dt, 512), cos=T(dt, Tk, 64), sin=T(dt, Tk, 64), wuk=T(dt, N, D, 512),
             kv_cache=kv, slot_mapping=T(I32, Tk), q_out=T(dt, Tk, N, 576 if mode == 0 else 512))
    if mode == 1:
        t.update(kv_cache_rope=T(dt, 192, 128, 1, 64), q_rope_out=T(dt, Tk, N, 64))
    t.update(kw)
    return t


def pp_code(tensors, mode=0, **scal):
    try:
        mla.mla_preprocess_workspace_size(tensors, 1e-6, cache_mode=mode, **scal)
        return 0
    except mla.MlaError as e:
        return e.code


def test_preprocess_valid_arguments(lib):
    assert pp_code(pp()) in (0, 361001)
    assert pp_code(pp(dt=F16)) in (0, 361001)
    assert pp_code(pp(mode=1), mode=1) in (0, 361001)
    assert pp_code(pp(bias0=None, bias1=None)) in (0, 361001)           # the biases are optional
    assert pp_code(pp(), do_rmsnorm=False) in (0, 361001)
    assert pp_code(pp(Tk=0)) == 0                                          # empty: no device query


def test_preprocess_nulls_and_patterns(lib):
    assert pp_code(pp(wuq=None)) == 161001
    assert pp_code(pp(mode=1, kv_cache_rope=None), mode=1) == 161001     # mode 1 needs the rope cache
    assert pp_code(pp(q_rope_out=T(BF16, 32, 128, 64))) == 161002        # mode 0 has no separate q^R
    t = pp()
    t["kv_cache_out"] = T(BF16, 192, 128, 1, 576)                           # not the same tensor as kvCache
    assert pp_code(t) == 161002
    assert pp_code(pp(ctkv_scale=T(BF16, 1))) == 161002                   # cacheMode 2 only


def test_preprocess_scalars(lib):
    assert pp_code(pp(), mode=2) == 161002                                  # NZ cache layouts are not built
    assert pp_code(pp(), mode=3) == 161002
    assert pp_code(pp(), quant_mode=1) == 161002
    assert pp_code(pp(), q_rope_dim=32) == 161002
    assert pp_code(pp(), q_rotary_coeff=4) == 161002
    assert pp_code(pp(), transpose_wuq=False) == 161002
    assert pp_code(pp(), wdkv_split_count=2) == 161002
    assert pp_code(pp(), wdq_dim=1024) == 161002


def test_preprocess_shapes_and_dtypes(lib):
    assert pp_code(pp(Tk=257)) == 161002                                    # tokenNum in [0, 256]
    assert pp_code(pp(gamma0=T(F16, 7168))) == 161002                       # every F tensor in the input's dtype
    assert pp_code(pp(wdqkv=T(BF16, 2112, 7168))) == 161002                 # int8 weights only (quantMode 0)
    assert pp_code(pp(de_scale0=T(F32, 2111))) == 161002
    assert pp_code(pp(slot_mapping=T(I64, 32))) == 161002                   # slotMapping is int32
    assert pp_code(pp(bias1=T(F32, 24576))) == 161002
    assert pp_code(pp(input=T(F32, 32, 7168))) == 161002
    assert pp_code(pp(wuk=T(BF16, 129, 128, 512), wuq=T(I8, 129 * 192, 1536), de_scale1=T(F32, 129 * 192),
                      bias1=T(I32, 129 * 192), q_out=T(BF16, 32, 129, 576))) == 161002   # headNum <= 128


def test_preprocess_tiling_rules(lib):
    Hcq = 1504                                                                # a multiple of 32, not of 64
    t = pp(wdqkv=T(I8, Hcq + 576, 7168), de_scale0=T(F32, Hcq + 576), bias0=T(I32, Hcq + 576),
           gamma1=T(BF16, Hcq), beta1=T(BF16, Hcq), wuq=T(I8, 128 * 192, Hcq))
    assert pp_code(t) == 561002
    D = 40                                                                    # not a multiple of 16
    t = pp(wuk=T(BF16, 128, D, 512), wuq=T(I8, 128 * (D + 64), 1536), de_scale1=T(F32, 128 * (D + 64)),
           bias1=T(I32, 128 * (D + 64)))
    assert pp_code(t) == 561002
    t = pp()
    t["input"].data = t["input"].data + 2
    assert pp_code(t) == 161002


def test_wait_probe_argument_checks(lib):
    import ctypes
    L = lib
    addr = ctypes.c_void_p(0x200000)   # never dereferenced: every case is rejected first
    assert L.mla_prolog_debug_wait_probe(None, 1024, 0, None) == 161001
    assert L.mla_prolog_debug_wait_probe(addr, 512, 0, None) == 161002      # shorter than the status word
    assert L.mla_prolog_debug_wait_probe(addr, 1024, 2, None) == 161002     # no such probe
    assert L.mla_prolog_debug_wait_probe(ctypes.c_void_p(0x200008), 1024, 0, None) == 161002   # misaligned


# ------------------------------------------------ the no-allocation entry point

def no_alloc_code(tensors, eps=1e-5, mode="PA_BSND"):
    return mla.mla_prolog_no_alloc(tensors, eps, eps, stream=0, cache_mode=mode, check=False)


def test_no_alloc_argument_checks(lib):
    """mla_prolog_no_alloc validates exactly like mla_prolog, before any CUDA call."""
    t = dsv3()
    t["w_uk"] = None
    assert no_alloc_code(t) == 161001
    t = dsv3()
    t["x"].data = None
    assert no_alloc_code(t) == 161001
    assert no_alloc_code(dsv3(w_dkvkr=T(BF16, 7168, 512))) == 161002
    assert no_alloc_code(dsv3(cache_index=T(F32, 32))) == 161002
    assert no_alloc_code(dsv3(q_out=T(I8, 32, 128, 512))) == 161001
    assert no_alloc_code(dsv3(), mode="PA_NZ") == 161002


def test_no_alloc_empty_tokens_returns_ok_without_the_device(lib):
    # T = 0: MLA_OK, and the call returns before it asks the runtime for anything
    t = dsv3(Tk=0, x=T(BF16, 0, 7168), rope_sin=T(BF16, 0, 64), rope_cos=T(BF16, 0, 64),
             cache_index=T(I64, 0), q_out=T(BF16, 0, 128, 512), q_rope_out=T(BF16, 0, 128, 64))
    assert no_alloc_code(t) == 0


def test_no_alloc_status_null_pointer(lib):
    assert lib.mla_prolog_no_alloc_status(None, None) == 161001
