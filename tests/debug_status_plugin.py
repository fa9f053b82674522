"""pytest plugin for runs against the debug build of the library
(GAR_LIBRARY=debug): before any comm is destroyed, its sticky device status
must still be AR_OK -- no device-side index check of any kernel launched on
it failed.  Loaded with ``-p debug_status_plugin`` by the debug-build test."""
import gradient_all_reduce_gb300 as gar

_destroy = gar.ar_destroy
checked = {"comms": 0}


def _checked_destroy(comm):
    status = gar.ar_get_async_error(comm)
    checked["comms"] += 1
    _destroy(comm)
    if status != gar.AR_OK:
        raise AssertionError(f"device status before ar_destroy: {gar.ar_status_string(status)}")


gar.ar_destroy = _checked_destroy


def pytest_sessionfinish(session, exitstatus):
    import re
    with open("/proc/self/maps") as f:
        maps = f.read()
    libs = sorted(set(re.findall(r"(libgar(?:_debug)?\.so)", maps)))
    print(f"\ndebug-build run: {checked['comms']} comms checked at destroy; loaded {libs}")
