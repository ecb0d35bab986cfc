"""pytest plugin for runs on the bounds-checked build: after the last test the
device error word must still be 0, i.e. no kernel access failed its bounds
test anywhere in the session.  Loaded with ``-p tests.status_plugin``."""


def pytest_sessionfinish(session, exitstatus):
    import zero_collectives_gb300 as zc
    code = zc.device_status()
    if code != 0:
        print(f"\ndevice error word {code} at the end of the session")
        session.exitstatus = 1
