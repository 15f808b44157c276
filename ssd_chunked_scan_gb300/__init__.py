"""GB300 (sm_103a) chunked SSD scan: a C-ABI CUDA library with a thin binding.

``ssd_chunked_scan_gb300.ssd`` is the binding (it loads libssd.so and raises
if it is missing); ``ssd_chunked_scan_gb300.inputs`` holds the seeded
synthetic workloads.  The binding is imported lazily so that the input
generators work on machines without the built library.
"""


def __getattr__(name):
    if name == "ssd_scan":
        from .autograd import ssd_scan
        return ssd_scan
    if name in ("ssd_fwd", "ssd_bwd", "ssd_fwd_ex", "ssd_bwd_ex", "ssd_set_path", "ssd_get_path", "ssd_strerror",
                "ssd_set_overlap", "ssd_get_overlap",
                "ssd_last_device_error", "SSDError", "SSD_PATH_TC", "SSD_PATH_SIMT"):
        from . import ssd
        return getattr(ssd, name)
    raise AttributeError(name)
