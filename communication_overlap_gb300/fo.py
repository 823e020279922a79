"""ctypes binding of libfo.so: the same function names as include/fo.h.

Argument marshalling only -- every step of the path runs in the library's
CUDA kernels.  Device buffers are passed as integer device addresses (for
example ``tensor.data_ptr()`` of a torch CUDA tensor) and streams as the raw
``cudaStream_t`` (``torch.cuda.Stream().cuda_stream``).  Loading fails
loudly if the library has not been built.
"""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libfo.so")

FO_OK, FO_ERR_ARG, FO_ERR_CUDA, FO_ERR_TIMEOUT, FO_ERR_UNSUPPORTED = range(5)
FO_NOALLOC_MAX_GROUPS = 4096   # include/fo.h
FO_LAYOUT_TILE, FO_LAYOUT_RS_SUBTILE, FO_LAYOUT_RS_ROWBLOCK, FO_LAYOUT_A2A_SUBTOKEN = range(4)
FO_CONS_COPY, FO_CONS_SUM, FO_CONS_RS, FO_CONS_A2A = range(4)
FO_GEMM_AUTO, FO_GEMM_SINGLE, FO_GEMM_PAIRS = range(3)
FO_ACT_NONE, FO_ACT_RELU, FO_ACT_SILU = range(3)
FO_BAND_FORWARD, FO_BAND_SERPENTINE = range(2)
FO_CONSUMER_SHARED, FO_CONSUMER_RESERVED = range(2)
(FO_TAB_SLOT_TILE, FO_TAB_TILE_SLOT, FO_TAB_SLOT_GROUP, FO_TAB_GROUP_TILES, FO_TAB_UNIT,
 FO_TAB_PART_START, FO_TAB_PART_LEN, FO_TAB_PART_DST, FO_TAB_DEST_UNITS,
 FO_TAB_FINAL_ROWS, FO_TAB_DEST_CAPACITY, FO_TAB_SLOT_LIVE, FO_TAB_UNIT_PLACE) = range(13)

_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p
_vpp = ctypes.POINTER(ctypes.c_void_p)
_dp = ctypes.POINTER(ctypes.c_double)


class fo_plan_desc(ctypes.Structure):
    _fields_ = [
        ("M", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
        ("swizzle", ctypes.c_int32), ("wave_width", ctypes.c_int32),
        ("n_groups", ctypes.c_int32), ("group_waves", _i32p),
        ("layout", ctypes.c_int32), ("n_dest", ctypes.c_int32),
        ("n_experts", ctypes.c_int32), ("expert_rows", _i32p),
        ("row_token", _i32p), ("row_slot", _i32p),
        ("host_only", ctypes.c_int32),
        ("pad_expert_tile_rows", ctypes.c_int32),
        ("band_order", ctypes.c_int32),
    ]


class FoError(RuntimeError):
    def __init__(self, call, status):
        self.status = status
        super().__init__(f"{call} failed: {fo_status_string(status)} ({status})")


_lib = None


def lib():
    """The loaded libfo.so (raises if it is missing: there is no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -m communication_overlap_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "fo_wave_count": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc), _i32p, _i32p]),
            "fo_plan_groups": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc), _vpp]),
            "fo_plan_info": (ctypes.c_int, [_vp, _i32p, _i32p, _i32p, _i32p, _i32p]),
            "fo_plan_table": (ctypes.c_int, [_vp, ctypes.c_int32, _i32p, ctypes.c_int64,
                                             ctypes.POINTER(ctypes.c_int64)]),
            "fo_plan_set_launch": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32,
                                                  ctypes.c_int32]),
            "fo_plan_set_trace": (ctypes.c_int, [_vp, _vp, _vp]),
            "fo_plan_set_pacing": (ctypes.c_int, [_vp, ctypes.c_int32]),
            "fo_plan_set_consumer_placement": (ctypes.c_int, [_vp, ctypes.c_int]),
            "fo_plan_set_gemm": (ctypes.c_int, [_vp, ctypes.c_int, _i32p, _i32p]),
            "fo_plan_set_split": (ctypes.c_int, [_vp, ctypes.c_int32, _i32p]),
            "fo_plan_device_status": (ctypes.c_int, [_vp, _i32p, ctypes.c_int32]),
            "fo_plan_destroy": (None, [_vp]),
            "fo_counting_table_init": (ctypes.c_int, [_vp, _vp, _vp]),
            "fo_signaled_gemm": (ctypes.c_int, [_vp, _vp, _vpp, _vp, _vp, _vp,
                                                ctypes.c_uint32, _vp]),
            "fo_consume_group": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int, _vp, _vpp,
                                                ctypes.c_int32, _vpp, _vp, ctypes.c_uint32,
                                                ctypes.c_uint64, _vp, _vp]),
            "fo_consume_group_noalloc": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int, _vp,
                                                        _vpp, ctypes.c_int32, _vpp, _vp,
                                                        ctypes.c_uint32, ctypes.c_uint64, _vp,
                                                        _vp]),
            "fo_reorder_back": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, _vpp,
                                               _vpp, _vp]),
            "fo_predict_partition": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc),
                                                    ctypes.c_double, _dp, _dp, ctypes.c_int32,
                                                    _dp]),
            "fo_tune_partition": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc), ctypes.c_double,
                                                 _dp, _dp, ctypes.c_int32, _i32p,
                                                 ctypes.c_int32, _i32p, _dp]),
            "fo_predict_partition_ex": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc),
                                                       ctypes.c_double, _dp, _dp, ctypes.c_int32,
                                                       ctypes.c_double, ctypes.c_double, _dp]),
            "fo_tune_partition_ex": (ctypes.c_int, [ctypes.POINTER(fo_plan_desc), ctypes.c_double,
                                                    _dp, _dp, ctypes.c_int32, ctypes.c_double,
                                                    ctypes.c_double, _i32p, ctypes.c_int32,
                                                    _i32p, _dp]),
            "fo_reorder_back_fused": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int32, _vpp,
                                                     _vpp, _vp, ctypes.c_int, _vp]),
            "fo_consume_reorder": (ctypes.c_int, [_vp, ctypes.c_int32, ctypes.c_int, _vp, _vpp,
                                                  ctypes.c_int32, _vpp, _vpp, _vp, ctypes.c_int,
                                                  _vp, ctypes.c_uint32, ctypes.c_uint64, _vp,
                                                  _vp]),
            "fo_allgather_rows": (ctypes.c_int, [_vp, _vpp, _vp, _vp, ctypes.c_int, _vp]),
            "fo_plan_route": (ctypes.c_int, [_vp, _vp, _vp, ctypes.c_int32, ctypes.c_int32,
                                             _vp, _vp]),
            "fo_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _ptrs(values):
    arr = (ctypes.c_void_p * max(1, len(values)))()
    for i, v in enumerate(values):
        arr[i] = int(v)
    return arr


def _i32(values):
    vals = [int(v) for v in values]
    return (ctypes.c_int32 * max(1, len(vals)))(*vals)


def _check(call, st):
    if st != FO_OK:
        raise FoError(call, st)


def fo_status_string(status):
    return lib().fo_status_string(int(status)).decode()


def make_desc(M, N, K, tile_m=128, tile_n=256, swizzle=8, wave_width=0,
              group_waves=(), layout=FO_LAYOUT_TILE, n_dest=1, expert_rows=None,
              row_token=None, row_slot=None, host_only=False, pad_expert_tile_rows=False,
              band_order=FO_BAND_FORWARD):
    """Build an fo_plan_desc; the returned object keeps its arrays alive."""
    d = fo_plan_desc()
    d.M, d.N, d.K = M, N, K
    d.tile_m, d.tile_n, d.swizzle, d.wave_width = tile_m, tile_n, swizzle, wave_width
    keep = []
    gw = _i32(group_waves)
    keep.append(gw)
    d.n_groups = len(group_waves)
    d.group_waves = ctypes.cast(gw, _i32p) if group_waves else None
    d.layout, d.n_dest = layout, n_dest
    if expert_rows is not None:
        er = _i32(expert_rows)
        keep.append(er)
        d.n_experts, d.expert_rows = len(expert_rows), ctypes.cast(er, _i32p)
    if row_token is not None:
        rt, rs = _i32(row_token), _i32(row_slot)
        keep += [rt, rs]
        d.row_token, d.row_slot = ctypes.cast(rt, _i32p), ctypes.cast(rs, _i32p)
    d.host_only = 1 if host_only else 0
    d.pad_expert_tile_rows = 1 if pad_expert_tile_rows else 0
    d.band_order = int(band_order)
    d._keep = keep
    return d


def fo_wave_count(desc):
    tiles, waves = ctypes.c_int32(), ctypes.c_int32()
    _check("fo_wave_count", lib().fo_wave_count(ctypes.byref(desc), ctypes.byref(tiles),
                                                ctypes.byref(waves)))
    return tiles.value, waves.value


def fo_plan_groups(desc):
    h = ctypes.c_void_p()
    _check("fo_plan_groups", lib().fo_plan_groups(ctypes.byref(desc), ctypes.byref(h)))
    return h.value


def fo_plan_info(plan):
    tiles, waves, P = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    _check("fo_plan_info", lib().fo_plan_info(plan, ctypes.byref(tiles), ctypes.byref(waves),
                                              ctypes.byref(P), None, None))
    gt = (ctypes.c_int32 * P.value)()
    ts = (ctypes.c_int32 * tiles.value)()
    _check("fo_plan_info", lib().fo_plan_info(plan, None, None, None, gt, ts))
    return tiles.value, waves.value, list(gt), list(ts)


def fo_plan_table(plan, which):
    n = ctypes.c_int64()
    _check("fo_plan_table", lib().fo_plan_table(plan, which, None, 0, ctypes.byref(n)))
    out = (ctypes.c_int32 * max(1, n.value))()
    _check("fo_plan_table", lib().fo_plan_table(plan, which, out, n.value, ctypes.byref(n)))
    return list(out)[:n.value]


def fo_plan_route(plan, row_token, row_slot, n_tokens, top_k, dev_status, stream):
    """Rebuild the All-to-All routing tables on the device from device int32
    arrays row_token[M], row_slot[M] (addresses), stream-ordered on `stream`."""
    _check("fo_plan_route", lib().fo_plan_route(plan, row_token, row_slot, n_tokens, top_k,
                                                dev_status, stream))


def fo_plan_set_launch(plan, consumer_ctas=0, reorder_ctas=0, overlap=True):
    _check("fo_plan_set_launch",
           lib().fo_plan_set_launch(plan, consumer_ctas, reorder_ctas, 1 if overlap else 0))


def fo_plan_set_pacing(plan, ctas_during_gemm=0):
    """Consumer CTAs that take work while the GEMM runs (0: all)."""
    _check("fo_plan_set_pacing", lib().fo_plan_set_pacing(plan, int(ctas_during_gemm)))


def fo_plan_set_consumer_placement(plan, placement=FO_CONSUMER_SHARED):
    """Consumer CTAs beside the GEMM's (shared) or only on the SMs the GEMM
    leaves free (reserved)."""
    _check("fo_plan_set_consumer_placement",
           lib().fo_plan_set_consumer_placement(plan, int(placement)))


def fo_plan_set_gemm(plan, variant=FO_GEMM_AUTO):
    """Select the GEMM variant; returns (pairs possible, pair capacity in CTAs)."""
    pairable, cap = ctypes.c_int32(), ctypes.c_int32()
    _check("fo_plan_set_gemm", lib().fo_plan_set_gemm(plan, variant, ctypes.byref(pairable),
                                                      ctypes.byref(cap)))
    return bool(pairable.value), cap.value


def fo_plan_set_split(plan, enable=True):
    """Enable or disable the last-wave split; returns the number of split tiles."""
    n = ctypes.c_int32()
    _check("fo_plan_set_split", lib().fo_plan_set_split(plan, 1 if enable else 0,
                                                        ctypes.byref(n)))
    return n.value


def fo_plan_set_trace(plan, stamps, consumer_stamps=0):
    """stamps: device uint64[tiles + W]; consumer_stamps: device
    uint64[2P + 4 * consumer CTAs]; 0 stops that trace."""
    _check("fo_plan_set_trace", lib().fo_plan_set_trace(plan, int(stamps) or None,
                                                        int(consumer_stamps) or None))


def fo_plan_device_status(plan, clear=False):
    st = ctypes.c_int32()
    _check("fo_plan_device_status",
           lib().fo_plan_device_status(plan, ctypes.byref(st), 1 if clear else 0))
    return st.value


def fo_plan_destroy(plan):
    if plan:
        lib().fo_plan_destroy(plan)


def fo_counting_table_init(plan, count, stream):
    _check("fo_counting_table_init",
           lib().fo_counting_table_init(plan, int(count), stream or None))


def fo_signaled_gemm(plan, A, B_list, C_r, count, flags, epoch, stream):
    """A, C_r, count, flags: device addresses (count/flags may be 0)."""
    _check("fo_signaled_gemm",
           lib().fo_signaled_gemm(plan, int(A), _ptrs(B_list), int(C_r), count or None,
                                  flags or None, epoch & 0xffffffff, stream or None))


def fo_consume_group(plan, group, kind, src, partials, dst, flags, epoch,
                     spin_limit_ns, dev_status, stream):
    _check("fo_consume_group",
           lib().fo_consume_group(plan, group, kind, int(src), _ptrs(partials),
                                  len(partials), _ptrs(dst), int(flags),
                                  epoch & 0xffffffff, spin_limit_ns, int(dev_status),
                                  stream or None))


def fo_consume_group_noalloc(plan, group, kind, src, partials, dst, flags, epoch,
                             spin_limit_ns, dev_status, stream):
    """fo_consume_group without any device allocation (fixed scratch inside
    the library; see include/fo.h)."""
    _check("fo_consume_group_noalloc",
           lib().fo_consume_group_noalloc(plan, group, kind, int(src), _ptrs(partials),
                                          len(partials), _ptrs(dst), int(flags),
                                          epoch & 0xffffffff, spin_limit_ns, int(dev_status),
                                          stream or None))


def fo_reorder_back(plan, group_begin, group_end, src, dst, stream):
    _check("fo_reorder_back",
           lib().fo_reorder_back(plan, group_begin, group_end, _ptrs(src), _ptrs(dst),
                                 stream or None))


def fo_reorder_back_fused(plan, group_begin, group_end, src, dst, bias, act, stream):
    """bias: device address of bf16[N] or 0."""
    _check("fo_reorder_back_fused",
           lib().fo_reorder_back_fused(plan, group_begin, group_end, _ptrs(src), _ptrs(dst),
                                       int(bias) or None, act, stream or None))


def fo_consume_reorder(plan, group, kind, src, partials, comm_dst, final_dst, bias, act,
                       flags, epoch, spin_limit_ns, dev_status, stream):
    """comm_dst: device addresses, or None for the direct variant (no
    communication buffers written)."""
    _check("fo_consume_reorder",
           lib().fo_consume_reorder(plan, group, kind, int(src), _ptrs(partials), len(partials),
                                    None if comm_dst is None else _ptrs(comm_dst),
                                    _ptrs(final_dst), int(bias) or None, act,
                                    int(flags), epoch & 0xffffffff, spin_limit_ns,
                                    int(dev_status), stream or None))


def fo_allgather_rows(plan, slices, out, bias, act, stream):
    _check("fo_allgather_rows",
           lib().fo_allgather_rows(plan, _ptrs(slices), int(out), int(bias) or None, act,
                                   stream or None))


def _curve(curve):
    pts = list(curve)
    b = (ctypes.c_double * len(pts))(*[float(x) for x, _ in pts])
    t = (ctypes.c_double * len(pts))(*[float(y) for _, y in pts])
    return b, t, len(pts)


def _factor(x):
    """An interference factor as passed to the library (None: 1)."""
    return 1.0 if x is None else float(x)


def fo_predict_partition(desc, gemm_us, curve, gemm_slowdown=None, comm_slowdown=None):
    """curve: [(bytes, us), ...]; desc carries the partition.  With either
    slowdown given, the interference model (fo_predict_partition_ex)."""
    b, t, n = _curve(curve)
    out = ctypes.c_double()
    if gemm_slowdown is None and comm_slowdown is None:
        _check("fo_predict_partition",
               lib().fo_predict_partition(ctypes.byref(desc), gemm_us, b, t, n,
                                          ctypes.byref(out)))
    else:
        _check("fo_predict_partition_ex",
               lib().fo_predict_partition_ex(ctypes.byref(desc), gemm_us, b, t, n,
                                             _factor(gemm_slowdown), _factor(comm_slowdown),
                                             ctypes.byref(out)))
    return out.value


def fo_tune_partition(desc, gemm_us, curve, gemm_slowdown=None, comm_slowdown=None):
    """Returns (waves per group, predicted us).  With either slowdown given,
    the interference model (fo_tune_partition_ex)."""
    b, t, n = _curve(curve)
    _, T = fo_wave_count(desc)
    parts = (ctypes.c_int32 * max(1, T))()
    ng = ctypes.c_int32()
    out = ctypes.c_double()
    if gemm_slowdown is None and comm_slowdown is None:
        _check("fo_tune_partition",
               lib().fo_tune_partition(ctypes.byref(desc), gemm_us, b, t, n, parts, T,
                                       ctypes.byref(ng), ctypes.byref(out)))
    else:
        _check("fo_tune_partition_ex",
               lib().fo_tune_partition_ex(ctypes.byref(desc), gemm_us, b, t, n,
                                          _factor(gemm_slowdown), _factor(comm_slowdown), parts,
                                          T, ctypes.byref(ng), ctypes.byref(out)))
    return list(parts)[:ng.value], out.value


def fo_predict_partition_ex(desc, gemm_us, curve, gemm_slowdown, comm_slowdown):
    """Algorithm 1's prediction with the interference factors."""
    return fo_predict_partition(desc, gemm_us, curve, gemm_slowdown, comm_slowdown)


def fo_tune_partition_ex(desc, gemm_us, curve, gemm_slowdown, comm_slowdown):
    """The exact search with the interference factors: (waves per group,
    predicted us)."""
    return fo_tune_partition(desc, gemm_us, curve, gemm_slowdown, comm_slowdown)


def partition_one_then_two(T):
    """Wave-group partition used by the workloads: one wave, then groups of
    two waves, the last group takes the remainder."""
    parts, left = [1], T - 1
    while left > 0:
        parts.append(min(2, left))
        left -= parts[-1]
    return parts
